// umma.cu — tensor-core (tcgen05) grouped GEMM for experts with many tokens.
//
// When a batch routes enough tokens to one expert (16 in a layer call or an
// explicit expert call; always the shared expert at batch >= 16), the
// expert's three matrices are a dense contraction: rows x K weights against
// K x tokens activations. Here the weights are dequantised (w = q*scale +
// bias, Flash-MoE page, "FMA Dequant") to fp16 in shared memory and
// tcgen05.mma (kind::f16, fp32 accumulation in tensor memory) multiplies them
// with the tokens' activations.
//
// Two kernels per matrix pair:
//  * k_tc_act stages every task's activations once per call as fp16 operand
//    tiles in global memory, already in the MMA's shared-memory layout (the
//    canonical no-swizzle K-major layout: 8x16-byte core matrices, the next
//    core matrix along K 128 bytes on, the next 8 rows 1024 bytes on), each
//    token scaled by a power of two that puts its largest magnitude in
//    [2^14, 2^15): fp16's range then holds any bf16 or fp32 input, and the
//    accumulators are scaled back exactly in the epilogue;
//  * k_tc_gemm streams each CTA's K range through a ring of 3-4 stages: the
//    weight codes and scale/bias rows arrive by TMA (cp.async.bulk.tensor on
//    3-D tensor maps of the expert pool, [expert][row][bytes]), the
//    activation tiles by bulk copy. The warps are specialised: one thread
//    copies, eight warps dequantise a step into one of 2-3 A tiles, one
//    thread issues the MMAs and commits them to mbarriers that free the stage
//    and the A tile, so copies, dequantisation and MMAs of successive steps
//    overlap.
// Within each 16-column block the columns are stored in the order the code
// extraction produces them (tc_slot); the activation tiles use the same order,
// so every dot product is unchanged.
//
// K is split over the CTAs of a thread-block cluster (one cluster per 128-row
// tile); the partial sums meet in distributed shared memory and are added in
// split order (deterministic). Every mbarrier wait is bounded (on expiry:
// BGQ_ERR_TIMEOUT in the status word, a bounded wait for the copies in
// flight, tensor memory freed, return); the cluster barriers are taken by
// every thread of every CTA on every path. The swizzled copies assume a
// 1024-byte aligned dynamic shared-memory base; a launch that does not get
// one writes BGQ_ERR_CUDA to the status word and computes nothing.
#include <cuda.h>

#include <mutex>
#include <vector>
#include <cuda_fp16.h>

#include "../../include/bgq.h"
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kTcWarps = 18;  // warp 0: copies, warp 1: MMAs, warps 2-17: dequantisation and epilogue
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcDq = 512;  // dequantising threads: four per weight row (a quarter K step each)
constexpr int kTcM = 128;
constexpr int kTcBK = 64;
constexpr long long kTcTimeoutNs = 1000000000ll;

__device__ __forceinline__ uint32_t tc_smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long tc_time() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tc_mbar_init(uint64_t* m, int count = 1) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem(m)), "r"(count) : "memory");
}
__device__ __forceinline__ void tc_arrive(uint64_t* m) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem(m)) : "memory");
}
__device__ __forceinline__ bool tc_mbar_try(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(tc_smem(m)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test, suspending the thread until the phase completes or
// kTcSuspendNs pass: waiting warps then leave the issue slots to the warps
// doing the work.
constexpr uint32_t kTcSuspendNs = 20000;
__device__ __forceinline__ bool tc_mbar_try_suspend(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(tc_smem(m)), "r"(parity), "r"(kTcSuspendNs)
      : "memory");
  return ok != 0;
}
// Bounded wait; false on timeout (the polling loop kept out of line).
__device__ __noinline__ bool tc_mbar_wait_loop(uint64_t* m, uint32_t parity, long long limit_ns) {
  const unsigned long long t0 = tc_time();
  long long it = 0;
  while (!tc_mbar_try_suspend(m, parity)) {
    if ((long long)(tc_time() - t0) > limit_ns || ++it > (1ll << 28)) return false;
  }
  return true;
}
__device__ __forceinline__ bool tc_mbar_wait(uint64_t* m, uint32_t parity, long long limit_ns) {
  return tc_mbar_try(m, parity) || tc_mbar_wait_loop(m, parity, limit_ns);
}
__device__ __forceinline__ void tc_fence_proxy() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Tensor memory: allocation and release by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major, no swizzle.
__device__ __forceinline__ uint64_t tc_desc(const void* base) {
  const uint64_t addr = (tc_smem(base) >> 4) & 0x3FFF;
  const uint64_t lbo = (128 >> 4);   // next core matrix along K
  const uint64_t sbo = (1024 >> 4);  // next 8 rows
  return addr | (lbo << 16) | (sbo << 32) | (1ull << 46);  // version 1, base offset 0, no swizzle
}
// Instruction descriptor: fp16 A and B (K-major), fp32 D, M = 128, N = n.
__device__ __forceinline__ uint32_t tc_idesc(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* m) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(tc_smem(m))
               : "memory");
}
// 8 consecutive fp32 columns of this warp's 32 tensor-memory lanes (one row per thread).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of element (row r, 16-column block kb, slot s in 0..15) in a
// K-major no-swizzle operand tile of 64 columns.
__device__ __forceinline__ int tc_off(int r, int kb, int s) {
  return (r >> 3) * 1024 + (kb * 2 + (s >> 3)) * 128 + (r & 7) * 16 + (s & 7) * 2;
}
// Slot of column k (0..15) inside its 16-column block, matching the order in
// which dequant_quarter() writes codes (4-bit: pairs (j, j+4) per 8 columns;
// 2-bit: pairs (j, j+8) per 16 columns).
template <int BITS>
__device__ __forceinline__ int tc_slot(int k) {
  if (BITS == 4) {
    const int h = k >> 3, j = k & 7;
    return h * 8 + (j < 4 ? 2 * j : 2 * (j - 4) + 1);
  } else {
    return k < 8 ? (k >> 2) * 8 + 2 * (k & 3) : ((k - 8) >> 2) * 8 + 2 * ((k - 8) & 3) + 1;
  }
}

// Dequantise quarter q (columns 16q..16q+15) of one row's 64 codes to fp16
// into the tile; qq points at that quarter's code words (2 at 4 bits, 1 at 2).
// fp16 1024 + code comes from placing the code under the exponent of 1024
// (0x6400); subtracting 1024 and one fused multiply-add give code*scale + bias.
template <int BITS>
__device__ __forceinline__ void dequant_quarter(const uint32_t* qq, uint32_t sbw, unsigned char* tile, int r, int q) {
  const __half2 s2 = __float2half2_rn(bf16lo(sbw));
  const __half2 b2 = __float2half2_rn(bf16hi(sbw));
  const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
  uint32_t w0, w1;
  if (BITS == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(qq);
    w0 = v.x;
    w1 = v.y;
  } else {
    w0 = w1 = *qq;
  }
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {  // chunk 2q + cc of the row: 8 codes
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // 4-bit: codes j and j+4 of word cc; 2-bit: codes 4cc+j and 4cc+j+8 of the word
      const uint32_t v = BITS == 4 ? ((cc ? w1 : w0) >> (4 * j)) & 0x000F000Fu : (w0 >> (2 * (4 * cc + j))) & 0x00030003u;
      const uint32_t m = v | 0x64006400u;
      __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&m), k1024);
      hh = __hfma2(hh, s2, b2);
      o[j] = *reinterpret_cast<uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(tile + tc_off(r, q, cc * 8)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------------------
// Copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_expect(uint64_t* m, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(m)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tc_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* m) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(tc_smem(dst)),
      "l"(src), "r"(bytes), "r"(tc_smem(m))
      : "memory");
}
// One box of a 3-D tensor map (x: byte within a row, y: row, z: expert).
__device__ __forceinline__ void tc_tma3(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* m) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(tc_smem(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(tc_smem(m))
      : "memory");
}

__device__ __forceinline__ void tc_fail(Ctrl* ctrl) { atomicExch(&ctrl->status, BGQ_ERR_TIMEOUT); }

constexpr int kTcMaxSplit = 8;   // K splits per tile: the CTAs of one cluster
constexpr int kTcMaxStages = 4;
constexpr int kTcChunk = 64;     // token columns per epilogue pass

// Cluster: barrier over every thread of every CTA (release / acquire), and
// loads from a peer CTA's shared memory.
__device__ __forceinline__ void tc_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t tc_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 tc_ld_peer4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Activation tiles: row pad_t + n of the staged activations holds token n of
// tensor-core task t (rows up to the task's token count rounded to 16 are
// zero). K step kb of every row lives in slab kb (rtot rows of 128 bytes).
// act_sh[row] = the power-of-two exponent the row was scaled by.
// One warp per row and 1024-column chunk (blockIdx.z): the row's largest
// magnitude (over the whole row), then the chunk's scaled fp16 values.
// ---------------------------------------------------------------------------
template <int BITS, bool F32>
__global__ void __launch_bounds__(256) k_tc_act(const Plan* __restrict__ plan, int B, int K,
                                                const void* __restrict__ src, int nslot, int kcols,
                                                unsigned char* __restrict__ act, int* __restrict__ act_sh, int rtot) {
  pdl_wait();     // the plan and src come from earlier kernels; act may still be read by one
  pdl_trigger();  // the GEMM behind this launch may start its prologue
  const int t = blockIdx.x;
  if (t >= (plan ? plan->nbig : 1)) return;
  const BigTask bt = plan ? plan_big(plan, B, K)[t] : BigTask{-1, B, 0, 0};
  const int npad = (bt.ntok + 15) & ~15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.y * 8 + warp;
  if (n >= npad) return;
  const int row = bt.pad + n;
  const bool live = n < bt.ntok;
  size_t srow = 0;
  if (live) {  // without a plan: token n, slot 0
    const int tok = plan ? plan_ptok(plan, B, K)[bt.first + n] : n;
    const int slot = plan ? plan_pslot(plan, B, K)[bt.first + n] : 0;
    srow = F32 ? ((size_t)tok * nslot + slot) * kcols : (size_t)tok * kcols;
  }
  auto load16 = [&](int b, float (&v)[16]) {
    if (!live) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    } else if (F32) {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + srow + b * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 a = p[i];
        v[4 * i] = a.x; v[4 * i + 1] = a.y; v[4 * i + 2] = a.z; v[4 * i + 3] = a.w;
      }
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + srow + b * 16);
      unpack_bf16x8(p[0], v);
      unpack_bf16x8(p[1], v + 8);
    }
  };
  const int nblk = kcols / 16;  // 16-column blocks of a row
  float m = 0.f;
  for (int b0 = lane; b0 < nblk; b0 += 32 * 4) {  // four blocks' loads in flight per lane
    float v[4][16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (b0 + 32 * u < nblk) {
        load16(b0 + 32 * u, v[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[u][i]));
  }
  m = warp_max(m);
  int sh = 0;  // the largest magnitude times 2^sh lands in [2^14, 2^15)
  if (m > 0.f) {
    const int e = (int)((__float_as_uint(m) >> 23) & 0xff) - 127;
    sh = 14 - e;
    sh = sh > 126 ? 126 : (sh < -126 ? -126 : sh);
  }
  if (lane == 0 && blockIdx.z == 0) act_sh[row] = sh;
  const float sc = exp2i(sh);
  const int b1 = min(nblk, ((int)blockIdx.z + 1) * 64);  // a chunk: two blocks per lane, both loaded first
  float v2[2][16];
#pragma unroll
  for (int u = 0; u < 2; ++u)
    if ((int)blockIdx.z * 64 + lane + 32 * u < b1) load16((int)blockIdx.z * 64 + lane + 32 * u, v2[u]);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int b = (int)blockIdx.z * 64 + lane + 32 * u;
    if (b >= b1) break;
    const float* v = v2[u];
    __half h[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) h[tc_slot<BITS>(k)] = __float2half_rn(v[k] * sc);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      w[k] = (uint32_t)__half_as_ushort(h[2 * k]) | ((uint32_t)__half_as_ushort(h[2 * k + 1]) << 16);
    unsigned char* tile = act + ((size_t)(b >> 2) * rtot + bt.pad) * 128;  // pad: a multiple of 16
    *reinterpret_cast<uint4*>(tile + tc_off(n, b & 3, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(tile + tc_off(n, b & 3, 8)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// ---------------------------------------------------------------------------
// The GEMM, one weight matrix of 128-row tiles. Gate/up (GU): tile t holds
// gate rows [64t, 64t+64) in its rows 0-63 and the same up rows in rows
// 64-127, so silu(gate) * up is formed where the tile's sums meet; down: 128
// rows of the down matrix.
// blockIdx.x = tile x nsplit K ranges (a cluster per tile), blockIdx.y = task.
// ---------------------------------------------------------------------------
struct TcMaps {
  CUtensorMap q[2][2];   // [routed pool, shared expert][gate or down, up]: codes, [expert][row][bytes]
  CUtensorMap sb[2][2];  // the matrices' scale/bias rows, same views
};
struct TcArgs {
  const Plan* plan;  // null: one task of every token (B tokens, slot 0) of the shared-expert view
  int B, K;
  int rows;        // output rows (f for gate/up, d for down)
  int y0[2][2];    // first row of matrix i in its map's expert region ([routed, shared][i])
  int kcols;       // input columns
  int nsplit;      // K splits = cluster size
  int g, stages, abufs;  // K steps per copy stage, copy stages, fp16 A tiles
  int sbw;               // scale/bias bytes per row and stage (32, or 16 for rows of 4 groups)
  const unsigned char* act;
  const int* act_sh;
  int rtot;
  float* out;      // H (gate/up) or Y (down), rows (token*nslot + slot)
  int nslot;
  uint16_t* y;     // down without a plan: bf16 output rows (token), in place of out when set
  float* yf;       // down without a plan: fp32 output rows (token), in place of out when set
  Ctrl* ctrl;
};

constexpr int kTcHead = 2048;  // barriers, tensor-memory address, flags, the tokens' unscale factors
constexpr int kTcSbBox = 32;   // scale/bias bytes per row and stage: the 8 groups from the stage's first aligned 4
// Shared memory of one CTA: head, `stages` copy stages (codes, scale/bias
// pairs, activation slabs of g K steps), `abufs` fp16 A tiles.
__host__ __device__ inline size_t tc_gemm_smem(int bits, int npad, int g, int stages, int abufs) {
  const size_t stage = (size_t)kTcM * g * (kTcBK * bits / 8) + kTcM * kTcSbBox + (size_t)g * npad * 128;
  return kTcHead + stages * stage + (size_t)abufs * kTcM * kTcBK * 2;
}

// One CTA: one tile over one K range; the cluster's CTAs (cluster rank = K
// split) cover the whole K. K step j lives in copy stage (j / g) % stages.
//   warp 0 (one thread): copies a stage's g K steps once the MMAs of the
//     stage's previous use have released it (codes and scale/bias by TMA,
//     activation slabs by bulk copy);
//   warps 2-17: dequantise step j's codes into A tile j % abufs (after the
//     MMAs of step j - abufs released it) and arrive on its `aready` barrier;
//   warp 1 (one thread): issues step j's MMAs once its A tile is complete,
//     commits them to the A tile's `afree` barrier and, at a stage's last
//     step, to the stage's `empty` barrier.
// Epilogue, per 64 token columns: every CTA copies its partial sums from
// tensor memory to shared memory; after a cluster barrier CTA r adds its
// share of the rows over every split in split order (deterministic), undoes
// the tokens' scales, applies silu(gate)*up (gate/up), stores.
template <int BITS, bool GU>
__global__ void __launch_bounds__(kTcThreads, 1) k_tc_gemm(const __grid_constant__ TcMaps maps, const TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int qb = kTcBK * BITS / 8;  // code bytes of one row and K step
  constexpr int kA = kTcM * kTcBK * 2;  // bytes of one fp16 A tile
  if (a.plan) pdl_wait();  // the plan comes from an earlier kernel (without one: after the barriers' set-up)
  if ((int)blockIdx.y >= (a.plan ? a.plan->nbig : 1)) return;  // the same for every CTA of a cluster
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tc_smem(smem) & 1023) {  // the swizzled copies need a 1024-byte aligned base (same for every CTA)
    if (tid == 0) atomicExch(&a.ctrl->status, BGQ_ERR_CUDA);
    return;
  }
  const BigTask bt = a.plan ? plan_big(a.plan, a.B, a.K)[blockIdx.y] : BigTask{-1, a.B, 0, 0};
  const int npad = (bt.ntok + 15) & ~15;
  const int tile = blockIdx.x / a.nsplit, split = blockIdx.x - tile * a.nsplit;
  const int G = a.g, S = a.stages, nA = a.abufs;
  const int cb = G * qb;                                  // code bytes of a row in one stage
  const int o_sb = kTcM * cb, o_act = o_sb + kTcM * a.sbw;
  const int stage_bytes = o_act + G * npad * 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [4] stage landed
  uint64_t* empty = full + kTcMaxStages;               // [4] stage read by its MMAs
  uint64_t* aready = empty + kTcMaxStages;             // [3] A tile dequantised
  uint64_t* afree = aready + 3;                        // [3] A tile read by its MMAs
  uint64_t* mdone = afree + 3;                         // every MMA complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mdone + 1);
  int* s_fail = reinterpret_cast<int*>(tslot + 1);
  float* s_un = reinterpret_cast<float*>(smem + 1024);  // [256] 2^-sh of each token
  unsigned char* stages = smem + kTcHead;
  unsigned char* atiles = stages + S * stage_bytes;  // [nA][kA]
  const int which = bt.expert < 0 ? 1 : 0, ez = bt.expert < 0 ? 0 : bt.expert;
  const int nkt = a.kcols / kTcBK;
  const int kb0 = nkt * split / a.nsplit, nk = nkt * (split + 1) / a.nsplit - kb0;
  const int nst = (nk + G - 1) / G;  // copy stages of this CTA's K range
  uint32_t ncols = 32;
  while ((int)ncols < npad) ncols <<= 1;
  if (tid == 0) {
    for (int i = 0; i < kTcMaxStages; ++i) {
      tc_mbar_init(&full[i]);
      tc_mbar_init(&empty[i]);
    }
    for (int i = 0; i < 3; ++i) {
      tc_mbar_init(&aready[i], kTcDq / 32);  // one arrival per dequantising warp
      tc_mbar_init(&afree[i]);
    }
    tc_mbar_init(mdone);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (!a.plan) pdl_wait();  // activations and their scales, written by the staging kernel
  pdl_trigger();
  // the copies start at once; warp 1 allocates tensor memory meanwhile
  if (warp == 0) {
    if (lane > 0)
      for (int n = lane - 1; n < npad; n += 31) s_un[n] = exp2i(-a.act_sh[bt.pad + n]);  // read in the epilogue
    if (lane == 0) {
      const bool sh = which == 1;
      const CUtensorMap* mq0 = sh ? &maps.q[1][0] : &maps.q[0][0];
      const CUtensorMap* mq1 = sh ? &maps.q[1][1] : &maps.q[0][1];
      const CUtensorMap* ms0 = sh ? &maps.sb[1][0] : &maps.sb[0][0];
      const CUtensorMap* ms1 = sh ? &maps.sb[1][1] : &maps.sb[0][1];
      const int y00 = sh ? a.y0[1][0] : a.y0[0][0], y01 = sh ? a.y0[1][1] : a.y0[0][1];
      // stage s = u % S and the parity of its previous use, kept incrementally
      // (no integer division in the per-step loops)
      int s = 0;
      uint32_t epar = 1;
      for (int u = 0, kb = kb0; u < nst; ++u, kb += G) {
        const int gs = min(G, nk - u * G);
        if (u >= S && !tc_mbar_wait(&empty[s], epar, kTcTimeoutNs)) {
          *s_fail = 1;
          break;
        }
        unsigned char* st = stages + s * stage_bytes;
        // a box is always copied whole (zero past the matrix's end)
        tc_expect(&full[s], (uint32_t)(o_act + gs * npad * 128));
        if (GU) {  // 64 gate rows, then the same 64 up rows
          const int y = tile * (kTcM / 2);
          tc_tma3(st, mq0, kb * qb, y00 + y, ez, &full[s]);
          tc_tma3(st + (kTcM / 2) * cb, mq1, kb * qb, y01 + y, ez, &full[s]);
          tc_tma3(st + o_sb, ms0, (kb >> 2) * 16, y00 + y, ez, &full[s]);
          tc_tma3(st + o_sb + (kTcM / 2) * a.sbw, ms1, (kb >> 2) * 16, y01 + y, ez, &full[s]);
        } else {
          const int y = y00 + tile * kTcM;
          tc_tma3(st, mq0, kb * qb, y, ez, &full[s]);
          tc_tma3(st + o_sb, ms0, (kb >> 2) * 16, y, ez, &full[s]);
        }
        for (int t = 0; t < gs; ++t)
          tc_bulk(st + o_act + t * npad * 128, a.act + ((size_t)(kb + t) * a.rtot + bt.pad) * 128,
                  (uint32_t)npad * 128, &full[s]);
        if (++s == S) {
          s = 0;
          epar ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    tmem_alloc(tslot, ncols);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    if (lane == 0) {
      const uint32_t idesc = tc_idesc(npad);
      int t = 0, s = 0, b = 0;  // step in stage, stage, A tile
      uint32_t fpar = 0, apar = 0;
      for (int j = 0; j < nk; ++j) {
        if (!tc_mbar_wait(&aready[b], apar, kTcTimeoutNs) || (t == 0 && !tc_mbar_wait(&full[s], fpar, kTcTimeoutNs))) {
          *s_fail = 1;
          break;
        }
        tc_fence_after();
        const unsigned char* bs = stages + s * stage_bytes + o_act + t * npad * 128;
        const unsigned char* at = atiles + b * kA;
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          tc_mma(tbase, tc_desc(at + kk * 256), tc_desc(bs + kk * 256), idesc, (j | kk) ? 1u : 0u);
        tc_commit(&afree[b]);
        if (t == G - 1 || j == nk - 1) tc_commit(&empty[s]);
        if (++b == nA) {
          b = 0;
          apar ^= 1;
        }
        if (++t == G) {
          t = 0;
          if (++s == S) {
            s = 0;
            fpar ^= 1;
          }
        }
      }
      tc_commit(mdone);  // tracks every MMA this thread issued
    }
  } else {
    // warp w of the 16 dequantises rows 8w..8w+7, lane l row 8w + l%8, quarter l/8
    const int e = tid - 64, rr = ((e >> 5) << 3) | (lane & 7), qt = lane >> 3;
    // the codes arrive swizzled (16-byte chunk c of row r at c ^ ((r*cb/128) % (cb/16)), cb >= 32)
    const int swz = cb >= 32 ? ((rr * cb) >> 7) & (cb / 16 - 1) : 0;
    int t = 0, s = 0, b = 0, ks = kb0 & ~3;  // step in stage, stage, A tile, the stage's first sb group
    uint32_t fpar = 0, apar = 0;
    for (int j = 0, kb = kb0; j < nk; ++j, ++kb) {
      // lane 0 waits for the stage and the A tile (freed by the MMAs of step j - nA), the warp follows
      int okw = 1;
      // (a stage's barrier completes once for all its steps: waited at its first)
      if (lane == 0)
        okw = (t > 0 || tc_mbar_wait(&full[s], fpar, kTcTimeoutNs)) &&
              (j < nA || tc_mbar_wait(&afree[b], apar ^ 1u, kTcTimeoutNs));
      if (!__shfl_sync(0xffffffffu, okw, 0)) {
        *s_fail = 1;
        break;
      }
      const unsigned char* st = stages + s * stage_bytes;
      const uint32_t sbw = *reinterpret_cast<const uint32_t*>(st + o_sb + rr * a.sbw + (kb - ks) * 4);
      const int x = t * qb + qt * (qb / 4);  // this quarter's first code byte in the row
      dequant_quarter<BITS>(reinterpret_cast<const uint32_t*>(st + rr * cb + ((((x >> 4) ^ swz) << 4) | (x & 15))), sbw,
                            atiles + b * kA, rr, qt);
      tc_fence_proxy();  // this thread's tile stores, visible to the tensor core
      __syncwarp();
      if (lane == 0) tc_arrive(&aready[b]);
      if (++b == nA) {
        b = 0;
        apar ^= 1;
      }
      if (++t == G) {
        t = 0;
        ks = (kb + 1) & ~3;
        if (++s == S) {
          s = 0;
          fpar ^= 1;
        }
      }
    }
  }
  // every MMA has completed before tensor memory is read (bounded)
  if (warp >= 2 && !tc_mbar_wait(mdone, 0, kTcTimeoutNs)) *s_fail = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool ok = *s_fail == 0;
  const uint32_t tbase = *tslot;
  if (!ok && tid == 0) {
    tc_fail(a.ctrl);
    // bounded waits for copies still in flight before the shared memory is released
    for (int i = 0; i < S; ++i) tc_mbar_wait(&full[i], 0, kTcTimeoutNs / 8) || tc_mbar_wait(&full[i], 1, 1000);
  }
  // epilogue (every CTA of the cluster takes the same passes and barriers)
  float* P = reinterpret_cast<float*>(stages);  // [kTcChunk tokens][128 rows] partial sums
  const uint32_t p_sa = tc_smem(P);
  const int orows = GU ? kTcM / 2 : kTcM;             // output rows of the tile
  const int rs = orows / a.nsplit, r0 = split * rs;  // this CTA's output rows of the reduction
  const int m0 = tile * orows;
  const size_t row_stride = (size_t)a.rows;
  const int* ptok = a.plan ? plan_ptok(a.plan, a.B, a.K) + bt.first : nullptr;  // null: token n, slot 0
  const int* pslot = a.plan ? plan_pslot(a.plan, a.B, a.K) + bt.first : nullptr;
  for (int c0 = 0; c0 < npad; c0 += kTcChunk) {
    const int cw = min(kTcChunk, npad - c0);
    if (ok && warp >= 2) {  // warp w reads tensor-memory lanes 32(w%4)..+31, a quarter (w-2)/4 of the columns
      const int sub = warp & 3, part = (warp - 2) >> 2;
      const int row = sub * 32 + lane;
      for (int c = part * 8; c < cw; c += 32) {
        float v[8];
        tmem_ld8(tbase + ((uint32_t)(sub * 32) << 16) + c0 + c, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) P[(c + k) * kTcM + row] = v[k];
      }
    }
    tc_cluster_sync();
    const int nq = rs / 4;  // row quads of this CTA
    for (int it = tid; it < cw * nq; it += kTcThreads) {
      const int c = it / nq, rq = r0 + 4 * (it - c * nq), n = c0 + c;
      if (!ok || n >= bt.ntok || m0 + rq >= a.rows) continue;
      const uint32_t off0 = p_sa + (uint32_t)((c * kTcM + rq) * 4);
      const uint32_t offu = off0 + (uint32_t)(kTcM / 2) * 4;  // the matching up rows (gate/up)
      // eight splits' loads in flight at once, each added in split order
      float4 g = make_float4(0.f, 0.f, 0.f, 0.f), w = g;
      for (int q0 = 0; q0 < a.nsplit; q0 += 8) {
        float4 gq[8], wq[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (q0 + k < a.nsplit) {
            gq[k] = tc_ld_peer4(tc_peer(off0, (uint32_t)(q0 + k)));
            if (GU) wq[k] = tc_ld_peer4(tc_peer(offu, (uint32_t)(q0 + k)));
          }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (q0 + k < a.nsplit) {
            g.x += gq[k].x; g.y += gq[k].y; g.z += gq[k].z; g.w += gq[k].w;
            if (GU) {
              w.x += wq[k].x; w.y += wq[k].y; w.z += wq[k].z; w.w += wq[k].w;
            }
          }
      }
      const float un = s_un[n];  // the token's scale, undone exactly
      float4 h;
      if (GU) {
        const float gx = g.x * un, gy = g.y * un, gz = g.z * un, gw = g.w * un;
        h.x = gx / (1.f + expf(-gx)) * (w.x * un);
        h.y = gy / (1.f + expf(-gy)) * (w.y * un);
        h.z = gz / (1.f + expf(-gz)) * (w.z * un);
        h.w = gw / (1.f + expf(-gw)) * (w.w * un);
      } else {
        h = make_float4(g.x * un, g.y * un, g.z * un, g.w * un);
      }
      if (!GU && (a.y || a.yf)) {  // one slot of weight 1: the combine's fma(1, y, 0), written here
        h = make_float4(__fadd_rn(h.x, 0.f), __fadd_rn(h.y, 0.f), __fadd_rn(h.z, 0.f), __fadd_rn(h.w, 0.f));
        const size_t o = (size_t)n * row_stride + m0 + rq;
        if (a.yf) *reinterpret_cast<float4*>(a.yf + o) = h;
        if (a.y)
          *reinterpret_cast<uint2*>(a.y + o) = make_uint2((uint32_t)f2bf(h.x) | ((uint32_t)f2bf(h.y) << 16),
                                                          (uint32_t)f2bf(h.z) | ((uint32_t)f2bf(h.w) << 16));
        continue;
      }
      const size_t orow = ptok ? (size_t)ptok[n] * a.nslot + pslot[n] : (size_t)n * a.nslot;
      *reinterpret_cast<float4*>(a.out + orow * row_stride + m0 + rq) = h;
    }
    tc_cluster_sync();  // peers are done reading before the next pass overwrites P (or the CTA exits)
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_free(tbase, ncols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int tc_npad_max(int B) {
  const int n = B < 256 ? B : 256;
  return (n + 15) & ~15;
}

// Clusters of n CTAs of this kernel the device can hold at once (asked once
// per device, kernel, shared-memory size and n).
static int tc_max_clusters(const void* kern, size_t smem, int n) {
  struct Entry {
    int dev;
    const void* kern;
    size_t smem;
    int n, count;
  };
  static std::mutex mu;
  static std::vector<Entry> seen;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : seen)
    if (e.dev == dev && e.kern == kern && e.smem == smem && e.n == n) return e.count;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)n;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int count = 0;
  if (cudaOccupancyMaxActiveClusters(&count, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    count = 0;
  }
  seen.push_back(Entry{dev, kern, smem, n, count});
  return count;
}

// K splits (the cluster size): the largest of 8, 4, 2 for which every tile's
// cluster is resident at once (no CTA waits for a second wave) and every CTA
// keeps at least two K steps; else 1.
static int tc_nsplit(const void* kern, size_t smem, int tiles, int kcols) {
  const int nkt = kcols / kTcBK;
  for (int n = kTcMaxSplit; n > 1; n >>= 1)
    if (n * 2 <= nkt && tiles <= tc_max_clusters(kern, smem, n)) return n;
  return 1;
}
// Pipeline shape within 227 KB of shared memory: the most K steps per copy
// stage (fewer, wider TMA boxes; at most the row's K steps), then the most
// stages, then A tiles.
static bool tc_pick(int bits, int npad, int nkt, int& g, int& stages, int& abufs) {
  for (int gg : {4, 2, 1})
    for (int ss : {3, 2})
      for (int aa : {3, 2})
        if (gg <= nkt && tc_gemm_smem(bits, npad, gg, ss, aa) <= 227 * 1024) {
          g = gg;
          stages = ss;
          abufs = aa;
          return true;
        }
  return false;
}
static size_t tc_up256(size_t n) { return (n + 255) & ~(size_t)255; }
// Rows of the staged activations: every task's tokens rounded up to 16.
int tc_act_rows(int B, int K) { return ((plan_max_pairs(B, K) + 15 * plan_max_big(B, K)) + 15) & ~15; }
size_t tc_act_bytes(int d, int f, int B, int K) {
  const int kc = d > f ? d : f;
  return tc_up256((size_t)tc_act_rows(B, K) * (kc / kTcBK) * 128) + tc_up256((size_t)tc_act_rows(B, K) * 4);
}

// cuTensorMapEncodeTiled, found through the runtime (the library does not link
// the driver library itself).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (EncodeTiledFn) nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A 3-D byte view [nexp][rows][row_bytes] of `base` (experts `estride` bytes
// apart), in boxes of box_bytes x box_rows rows x 1 expert.
static bool make_map(CUtensorMap* m, const void* base, int row_bytes, int rows, int nexp, long long estride,
                     int box_bytes, int box_rows, bool swizzle = false) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc || !base || (uintptr_t)base % 16 || row_bytes % 16 || estride % 16 || box_bytes % 16) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)rows, (cuuint64_t)nexp};
  const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)estride};
  const cuuint32_t box[3] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  // swizzled: the box's 16-byte chunks XOR-permuted over the box width (32, 64 or 128 bytes)
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle && box_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (swizzle && box_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle && box_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the gate/up (gu) or down matrices of the routed pool and the
// shared expert, in boxes of g K steps (codes) or sbw bytes (scale/bias)
// by 64 (gate/up) or 128 (down) rows. y0 receives each matrix's first row in
// its map's expert region.
static bool tc_maps(const ExpertSet& es, bool gu, int g, int sbw, TcMaps& M, int (&y0)[2][2]) {
  const int d = es.d, f = es.f, bits = es.bits;
  const int kc = gu ? d : f, rows = gu ? f : d;
  const int rb = kc * bits / 8, sbb = (kc / kGroup) * 4, qb = g * kTcBK * bits / 8;
  const int br = gu ? kTcM / 2 : kTcM;
  const long long mw = (long long)d * f * bits / 32, mg = (long long)d * f / kGroup * 2;
  memset(&M, 0, sizeof(M));
  // the shared expert (or the one explicit expert): each matrix its own view
  const void* sq[2] = {gu ? (const void*)es.shared.gate_q : (const void*)es.shared.down_q,
                       (const void*)es.shared.up_q};
  const void* ss[2] = {gu ? (const void*)es.shared.gate_sb : (const void*)es.shared.down_sb,
                       (const void*)es.shared.up_sb};
  for (int i = 0; i < (gu ? 2 : 1); ++i) {
    if (!make_map(&M.q[1][i], sq[i], rb, rows, 1, (long long)rb * rows, qb, br, true)) return false;
    if (!make_map(&M.sb[1][i], ss[i], sbb, rows, 1, (long long)sbb * rows, sbw, br)) return false;
    y0[1][i] = 0;
  }
  if (!es.pool_q) {  // no routed pool: never used
    M.q[0][0] = M.q[1][0];
    M.sb[0][0] = M.sb[1][0];
    M.q[0][1] = M.q[1][gu ? 1 : 0];
    M.sb[0][1] = M.sb[1][gu ? 1 : 0];
    y0[0][0] = y0[0][1] = 0;
    return true;
  }
  // the routed pool: one view per matrix kind over every expert; gate/up
  // rows f apart in an expert's region of 3f rows of d columns
  const char* pq = reinterpret_cast<const char*>(es.pool_q) + (gu ? 0 : 2 * mw * 4);
  const char* ps = reinterpret_cast<const char*>(es.pool_sb) + (gu ? 0 : 2 * mg * 2);
  const int region = gu ? 3 * f : d;
  // nexp: enough experts to cover any index the plan can name (the pool's rows are all in range)
  const int nexp = 1024;
  if (!make_map(&M.q[0][0], pq, rb, region, nexp, es.q_stride * 4, qb, br, true)) return false;
  if (!make_map(&M.sb[0][0], ps, sbb, region, nexp, es.sb_stride * 2, sbw, br)) return false;
  M.q[0][1] = M.q[0][0];
  M.sb[0][1] = M.sb[0][0];
  y0[0][0] = 0;
  y0[0][1] = gu ? f : 0;
  return true;
}

// Whether a layer's pools can feed the tensor-core path (tensor-map alignment).
bool tc_layer_ok(const ExpertSet& es) {
  TcMaps M;
  int y0[2][2];
  return encode_tiled() != nullptr && tc_maps(es, true, 1, 16, M, y0) && tc_maps(es, false, 1, 16, M, y0);
}

template <int BITS>
static cudaError_t tc_run(const ExpertSet& es, bool gu, const Plan* plan, int B, int K, const void* src, float* out,
                          int nslot, Ctrl* ctrl, unsigned char* act, uint16_t* y, float* yf, cudaStream_t s) {
  TcArgs a{};
  const int nbig_max = plan ? plan_max_big(B, K) : 1;
  const int npad = tc_npad_max(B);
  const int kc = gu ? es.d : es.f;
  if (!tc_pick(BITS, npad, kc / kTcBK, a.g, a.stages, a.abufs)) return cudaErrorInvalidValue;
  a.sbw = (kc / kGroup) * 4 >= kTcSbBox ? kTcSbBox : 16;  // a box never wider than the row
  TcMaps M;
  if (!tc_maps(es, gu, a.g, a.sbw, M, a.y0)) return cudaErrorInvalidValue;
  a.plan = plan;
  a.B = B;
  a.K = K;
  a.rows = gu ? es.f : es.d;
  a.kcols = gu ? es.d : es.f;
  a.rtot = tc_act_rows(B, K);
  a.act = act;
  a.act_sh = reinterpret_cast<const int*>(act + tc_up256((size_t)a.rtot * (((es.d > es.f ? es.d : es.f)) / kTcBK) * 128));
  a.out = out;
  a.nslot = nslot;
  a.y = y;
  a.yf = yf;
  a.ctrl = ctrl;
  int* act_sh = const_cast<int*>(a.act_sh);
  // Both launches are programmatic dependents of the kernel before them on
  // the stream (each waits for it before touching memory it shares), so a
  // launch's set-up overlaps the previous kernel's tail: an explicit expert
  // call at 16 / 64 tokens took 31.0 / 33.2 us without, 27.1 / 30.2 us with.
  // Not at 256 tokens (52.8 us without, 54.0 us with).
  const bool overlap = npad <= 128;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  // stage the activations once
  cudaLaunchConfig_t ca = {};
  ca.gridDim = dim3(nbig_max, (npad + 7) / 8, (a.kcols + 1023) / 1024);
  ca.blockDim = dim3(256);
  ca.stream = s;
  ca.attrs = at;
  ca.numAttrs = 1;
  const int rt = a.rtot;  // kc == a.kcols
  cudaError_t e = gu ? cudaLaunchKernelEx(&ca, k_tc_act<BITS, false>, plan, B, K, src, nslot, kc, act, act_sh, rt)
                     : cudaLaunchKernelEx(&ca, k_tc_act<BITS, true>, plan, B, K, src, nslot, kc, act, act_sh, rt);
  if (e != cudaSuccess) return e;
  const size_t sm = tc_gemm_smem(BITS, npad, a.g, a.stages, a.abufs);
  void* kern = gu ? (void*)k_tc_gemm<BITS, true> : (void*)k_tc_gemm<BITS, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int tiles = gu ? (a.rows + kTcM / 2 - 1) / (kTcM / 2) : (a.rows + kTcM - 1) / kTcM;
  a.nsplit = tc_nsplit(kern, sm, tiles, a.kcols);
  // one cluster per tile and task: its CTAs are the tile's K splits
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * a.nsplit, nbig_max);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = (unsigned)a.nsplit;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (gu) return cudaLaunchKernelEx(&cfg, k_tc_gemm<BITS, true>, M, a);
  return cudaLaunchKernelEx(&cfg, k_tc_gemm<BITS, false>, M, a);
}

cudaError_t launch_gateup_tc(const ExpertSet& es, const Plan* plan, int B, int K, const uint16_t* x, float* H,
                             int nslot, Ctrl* ctrl, unsigned char* act, cudaStream_t s) {
  if (B < kBigTok) return cudaSuccess;  // no task can have 16 tokens
  return es.bits == 4 ? tc_run<4>(es, true, plan, B, K, x, H, nslot, ctrl, act, nullptr, nullptr, s)
                      : tc_run<2>(es, true, plan, B, K, x, H, nslot, ctrl, act, nullptr, nullptr, s);
}

cudaError_t launch_down_tc(const ExpertSet& es, const Plan* plan, int B, int K, const float* H, float* Y, int nslot,
                           Ctrl* ctrl, unsigned char* act, uint16_t* y, float* y_f32, cudaStream_t s) {
  if (B < kBigTok) return cudaSuccess;
  if ((y || y_f32) && plan) return cudaErrorInvalidValue;  // direct output: the one-task form only
  return es.bits == 4 ? tc_run<4>(es, false, plan, B, K, H, Y, nslot, ctrl, act, y, y_f32, s)
                      : tc_run<2>(es, false, plan, B, K, H, Y, nslot, ctrl, act, y, y_f32, s);
}

}  // namespace bgq
