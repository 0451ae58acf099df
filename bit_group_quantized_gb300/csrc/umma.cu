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
//    activation tiles by bulk copy; the CTA's 256 threads dequantise a step
//    into one of two A tiles while the tensor core multiplies the previous
//    one; one thread issues the MMAs and commits them to mbarriers that free
//    the stage and the A tile.
// Within each 16-column block the columns are stored in the order the code
// extraction produces them (tc_slot); the activation tiles use the same order,
// so every dot product is unchanged.
//
// K is split over several CTAs per 128-row tile; the tile's last CTA adds the
// fp32 partial sums in split order (deterministic). Every wait is bounded
// (on expiry: BGQ_ERR_TIMEOUT in the status word, a bounded wait for the
// copies and MMAs in flight, tensor memory freed, return).
#include <cuda.h>
#include <cuda_fp16.h>

#include "../../include/bgq.h"
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kTcThreads = 256;  // two threads per weight row (half a K step each)
constexpr int kTcM = 128;
constexpr int kTcBK = 64;
constexpr long long kTcTimeoutNs = 1000000000ll;

__device__ __forceinline__ uint32_t tc_smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long tc_time() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tc_mbar_init(uint64_t* m) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(m)) : "memory");
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
// Bounded wait; false on timeout.
__device__ bool tc_mbar_wait(uint64_t* m, uint32_t parity, long long limit_ns) {
  if (tc_mbar_try(m, parity)) return true;
  const unsigned long long t0 = tc_time();
  long long it = 0;
  while (!tc_mbar_try(m, parity)) {
    if ((++it & 63) == 0 && ((long long)(tc_time() - t0) > limit_ns || it > (1ll << 28))) return false;
  }
  return true;
}
__device__ __forceinline__ void tc_fence_proxy() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Asynchronous global -> shared copies (16 bytes through L2 only, 4 bytes), grouped per K step.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc_smem(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(tc_smem(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc_smem(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
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
// which dequant_half() writes codes (4-bit: pairs (j, j+4) per 8 columns;
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

// Dequantise half h (columns 32h..32h+31) of one row's 64 codes to fp16 into
// the tile; qh points at that half's code words (4 at 4 bits, 2 at 2 bits).
template <int BITS>
__device__ __forceinline__ void dequant_half(const uint32_t* qh, uint32_t sbw, unsigned char* tile, int r, int h) {
  const __half2 s2 = __float2half2_rn(bf16lo(sbw));
  const __half2 b2 = __float2half2_rn(bf16hi(sbw));
  const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
  uint32_t w[4];
  if (BITS == 4) {
    const uint4 a = *reinterpret_cast<const uint4*>(qh);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(qh);
    w[0] = a.x; w[1] = a.y; w[2] = 0; w[3] = 0;
  }
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * h + cc;  // chunk of the row
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v;
      if (BITS == 4) {
        v = (w[cc] >> (4 * j)) & 0x000F000Fu;  // codes j and j+4 of word c
      } else {
        const int base = (cc & 1) * 4;                    // chunk c: half (c&1) of word c/2
        v = (w[cc >> 1] >> (2 * (base + j))) & 0x00030003u;  // codes base+j and base+j+8
      }
      const uint32_t m = v | 0x64006400u;
      __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&m), k1024);
      hh = __hfma2(hh, s2, b2);
      o[j] = *reinterpret_cast<uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(tile + tc_off(r, c >> 1, (c & 1) * 8)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}


// Write 16 activation values (columns 16*kb .. +15 of token row n) into the
// tile in tc_slot order.
template <int BITS>
__device__ __forceinline__ void put_act16(unsigned char* tile, int n, int kb, const float (&v)[16]) {
  __half h[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) h[tc_slot<BITS>(k)] = __float2half_rn(v[k]);
  uint4 c0, c1;
  c0.x = (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
  c0.y = (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16);
  c0.z = (uint32_t)__half_as_ushort(h[4]) | ((uint32_t)__half_as_ushort(h[5]) << 16);
  c0.w = (uint32_t)__half_as_ushort(h[6]) | ((uint32_t)__half_as_ushort(h[7]) << 16);
  c1.x = (uint32_t)__half_as_ushort(h[8]) | ((uint32_t)__half_as_ushort(h[9]) << 16);
  c1.y = (uint32_t)__half_as_ushort(h[10]) | ((uint32_t)__half_as_ushort(h[11]) << 16);
  c1.z = (uint32_t)__half_as_ushort(h[12]) | ((uint32_t)__half_as_ushort(h[13]) << 16);
  c1.w = (uint32_t)__half_as_ushort(h[14]) | ((uint32_t)__half_as_ushort(h[15]) << 16);
  *reinterpret_cast<uint4*>(tile + tc_off(n, kb, 0)) = c0;
  *reinterpret_cast<uint4*>(tile + tc_off(n, kb, 8)) = c1;
}

__device__ __forceinline__ ExpertRef tc_resolve(const ExpertSet& es, int e) {
  if (e < 0) return es.shared;
  ExpertRef r;
  const long long mw = (long long)es.d * es.f * es.bits / 32;
  const long long mg = (long long)es.d * es.f / kGroup * 2;
  const uint32_t* q = es.pool_q + (long long)e * es.q_stride;
  const uint16_t* sb = es.pool_sb + (long long)e * es.sb_stride;
  r.gate_q = q;
  r.up_q = q + mw;
  r.down_q = q + 2 * mw;
  r.gate_sb = sb;
  r.up_sb = sb + mg;
  r.down_sb = sb + 2 * mg;
  return r;
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

constexpr int kTcMaxSplit = 8;  // K splits per tile (partial sums reduced by the tile's last CTA)
constexpr int kTcMaxStages = 4;

// Split K: every CTA of a tile publishes its partial sums, then counts itself
// in *cnt; true (for the whole block) in the last one, which resets *cnt for
// the next launch. Nothing waits, so a failed CTA cannot hang the others.
__device__ bool tc_last_of_tile(int* cnt, int nsplit) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(cnt, 1);
    s_last = prev == nsplit - 1;
    if (s_last) *cnt = 0;
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last != 0;
}

// ---------------------------------------------------------------------------
// Activation tiles: row pad_t + n of the staged activations holds token n of
// tensor-core task t (rows up to the task's token count rounded to 16 are
// zero). K step kb of every row lives in slab kb (rtot rows of 128 bytes).
// act_sh[row] = the power-of-two exponent the row was scaled by.
// One warp per row: the row's largest magnitude, then its scaled fp16 values.
// ---------------------------------------------------------------------------
template <int BITS, bool F32>
__global__ void __launch_bounds__(256) k_tc_act(const Plan* __restrict__ plan, int B, int K,
                                                const void* __restrict__ src, int nslot, int kcols,
                                                unsigned char* __restrict__ act, int* __restrict__ act_sh, int rtot) {
  const int t = blockIdx.x;
  if (t >= plan->nbig) return;
  const BigTask bt = plan_big(plan, B, K)[t];
  const int npad = (bt.ntok + 15) & ~15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.y * 8 + warp;
  if (n >= npad) return;
  const int row = bt.pad + n;
  const bool live = n < bt.ntok;
  size_t srow = 0;
  if (live) {
    const int tok = plan_ptok(plan, B, K)[bt.first + n];
    srow = F32 ? ((size_t)tok * nslot + plan_pslot(plan, B, K)[bt.first + n]) * kcols : (size_t)tok * kcols;
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
  for (int b = lane; b < nblk; b += 32) {
    float v[16];
    load16(b, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  m = warp_max(m);
  int sh = 0;  // the largest magnitude times 2^sh lands in [2^14, 2^15)
  if (m > 0.f) {
    const int e = (int)((__float_as_uint(m) >> 23) & 0xff) - 127;
    sh = 14 - e;
    sh = sh > 126 ? 126 : (sh < -126 ? -126 : sh);
  }
  if (lane == 0) act_sh[row] = sh;
  const float sc = exp2i(sh);
  for (int b = lane; b < nblk; b += 32) {
    float v[16];
    load16(b, v);
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
// The GEMM. NA = 2: gate and up (silu(gate) * up); NA = 1: down.
// blockIdx.x = 128-row tile x nsplit K ranges, blockIdx.y = tensor-core task.
// ---------------------------------------------------------------------------
struct TcMaps {
  CUtensorMap q[2][2];   // [routed pool, shared expert][matrix]: codes, [expert][row][bytes]
  CUtensorMap sb[2][2];  // the matrices' scale/bias rows, same views
};
struct TcArgs {
  const Plan* plan;
  int B, K;
  int rows;        // output rows of each matrix
  int y0[2][2];    // first row of matrix i in its map's expert region ([routed, shared][i])
  int kcols;       // input columns
  int nsplit;
  const unsigned char* act;
  const int* act_sh;
  int rtot;
  float* out;      // H (gate/up) or Y (down), rows (token*nslot + slot)
  int nslot;
  Ctrl* ctrl;
  float* part;
  int* cnt;
};

__host__ __device__ inline int tc_stages(int npad) { return npad <= 128 ? 4 : 3; }
__host__ __device__ inline size_t tc_gemm_smem(int na, int bits, int npad) {
  const int stage = na * kTcM * (kTcBK * bits / 8) + npad * 128;
  return 1024 + (size_t)tc_stages(npad) * stage + 2 * na * kTcM * 16 + 2 * na * kTcM * kTcBK * 2;
}

template <int BITS, int NA>
__global__ void __launch_bounds__(kTcThreads, 1) k_tc_gemm(const __grid_constant__ TcMaps maps, const TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int qb = kTcBK * BITS / 8;  // code bytes of one row and K step
  constexpr int kA = kTcM * kTcBK * 2;  // bytes of one fp16 A tile
  if ((int)blockIdx.y >= a.plan->nbig) return;
  const BigTask bt = plan_big(a.plan, a.B, a.K)[blockIdx.y];
  const int npad = (bt.ntok + 15) & ~15;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int tile = blockIdx.x / a.nsplit, split = blockIdx.x - tile * a.nsplit;
  const int m0 = tile * kTcM;
  const int S = tc_stages(npad);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [4] stage landed
  uint64_t* empty = full + kTcMaxStages;               // [4] stage read by its MMAs
  uint64_t* adone = empty + kTcMaxStages;              // [2] A tile read by its MMAs
  uint32_t* tslot = reinterpret_cast<uint32_t*>(adone + 2);
  int* s_fail = reinterpret_cast<int*>(tslot + 1);
  const int stage_bytes = NA * kTcM * qb + npad * 128;
  unsigned char* stages = smem + 1024;
  unsigned char* sbring = stages + S * stage_bytes;       // [2 groups of 4 K steps][NA][128 rows][16 B]
  unsigned char* atiles = sbring + 2 * NA * kTcM * 16;    // [2][NA][kA]
  const int which = bt.expert < 0 ? 1 : 0, ez = bt.expert < 0 ? 0 : bt.expert;
  const int nkt = a.kcols / kTcBK;
  const int kb0 = nkt * split / a.nsplit, nk = nkt * (split + 1) / a.nsplit - kb0;
  uint32_t ncols = 32;
  while ((int)ncols < NA * npad) ncols <<= 1;
  if (tid == 0) {
    for (int i = 0; i < kTcMaxStages; ++i) {
      tc_mbar_init(&full[i]);
      tc_mbar_init(&empty[i]);
    }
    tc_mbar_init(&adone[0]);
    tc_mbar_init(&adone[1]);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t idesc = tc_idesc(npad);
  // thread 0: K step kb0 + j into stage j % S (scale/bias rows of four K
  // steps at a time, at the first step of each group in the range)
  auto issue = [&](int j) {
    const int kb = kb0 + j, s = j % S;
    unsigned char* st = stages + s * stage_bytes;
    const bool with_sb = j == 0 || (kb & 3) == 0;
    tc_expect(&full[s], (uint32_t)(NA * kTcM * qb + npad * 128 + (with_sb ? NA * kTcM * 16 : 0)));
#pragma unroll
    for (int i = 0; i < NA; ++i) {
      const int y = a.y0[which][i] + m0;
      tc_tma3(st + i * kTcM * qb, &maps.q[which][i], kb * qb, y, ez, &full[s]);
      if (with_sb) tc_tma3(sbring + (((kb >> 2) & 1) * NA + i) * kTcM * 16, &maps.sb[which][i], (kb >> 2) * 16, y, ez,
                           &full[s]);
    }
    tc_bulk(st + NA * kTcM * qb, a.act + ((size_t)kb * a.rtot + bt.pad) * 128, (uint32_t)npad * 128, &full[s]);
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < S - 1 && issued < nk; ++issued) issue(issued);
  const int rr = tid & (kTcM - 1), hf = tid >> 7;  // the row this thread dequantises, and which half of its codes
  int j = 0;
  for (; j < nk; ++j) {
    const int kb = kb0 + j, s = j % S;
    if (tid == 0 && issued < nk) {
      // the stage of step j + S - 1 was last read by the MMAs of step j - 1
      if (j >= 1 && !tc_mbar_wait(&empty[(j - 1) % S], (uint32_t)(((j - 1) / S) & 1), kTcTimeoutNs)) *s_fail = 1;
      else issue(issued++);
    }
    if (!tc_mbar_wait(&full[s], (uint32_t)((j / S) & 1), kTcTimeoutNs)) *s_fail = 1;
    if (j >= 2 && !tc_mbar_wait(&adone[j & 1], (uint32_t)(((j - 2) >> 1) & 1), kTcTimeoutNs)) *s_fail = 1;
    const unsigned char* st = stages + s * stage_bytes;
    unsigned char* at = atiles + (j & 1) * NA * kA;
#pragma unroll
    for (int i = 0; i < NA; ++i) {
      const uint32_t sbw =
          *reinterpret_cast<const uint32_t*>(sbring + (((kb >> 2) & 1) * NA + i) * kTcM * 16 + rr * 16 + (kb & 3) * 4);
      dequant_half<BITS>(reinterpret_cast<const uint32_t*>(st + i * kTcM * qb + rr * qb + hf * (qb / 2)), sbw,
                         at + i * kA, rr, hf);
    }
    tc_fence_proxy();
    __syncthreads();
    if (*s_fail) break;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTcBK / 16; ++kk) {
        const uint64_t bd = tc_desc(st + NA * kTcM * qb + kk * 256);
#pragma unroll
        for (int i = 0; i < NA; ++i)
          tc_mma(tbase + i * npad, tc_desc(at + i * kA + kk * 256), bd, idesc, (j | kk) ? 1u : 0u);
      }
      tc_commit(&adone[j & 1]);
      tc_commit(&empty[s]);
    }
  }
  bool ok = *s_fail == 0;
  // the last commit covers every MMA
  if (ok && !tc_mbar_wait(&adone[(nk - 1) & 1], (uint32_t)(((nk - 1) >> 1) & 1), kTcTimeoutNs)) ok = false;
  const size_t pc = (size_t)plan_max_pairs(a.B, a.K);
  const int* ptok = plan_ptok(a.plan, a.B, a.K) + bt.first;
  const int* pslot = plan_pslot(a.plan, a.B, a.K) + bt.first;
  if (ok && warp < 4) {  // warp w reads tensor-memory lanes 32w..32w+31
    tc_fence_after();
    const int row = m0 + warp * 32 + (tid & 31);
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int c0 = 0; c0 < npad; c0 += 8) {
      float acc[NA][8];
#pragma unroll
      for (int i = 0; i < NA; ++i) tmem_ld8(tbase + lane_off + i * npad + c0, acc[i]);
      if (row < a.rows) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int n = c0 + u;
          if (n >= bt.ntok) continue;
          const float un = exp2i(-a.act_sh[bt.pad + n]);  // the token's scale, undone exactly
          if (NA == 2) {
            const float g = acc[0][u] * un, up = acc[NA - 1][u] * un;
            if (a.nsplit == 1) {
              a.out[((size_t)ptok[n] * a.nslot + pslot[n]) * a.rows + row] = g / (1.f + expf(-g)) * up;
            } else {  // partial sums of this K range: [split][pair][gate, up][row]
              float* pp = a.part + (((size_t)split * pc + bt.first + n) * 2) * a.rows + row;
              pp[0] = g;
              pp[a.rows] = up;
            }
          } else {
            const float y = acc[0][u] * un;
            if (a.nsplit == 1)
              a.out[((size_t)ptok[n] * a.nslot + pslot[n]) * a.rows + row] = y;
            else  // [split][pair][row]
              a.part[((size_t)split * pc + bt.first + n) * a.rows + row] = y;
          }
        }
      }
    }
  } else if (!ok && tid == 0) {
    tc_fail(a.ctrl);
    // bounded waits for the copies and MMAs in flight before the memory is released
    for (int i = 0; i < S; ++i) tc_mbar_wait(&full[i], 0, kTcTimeoutNs / 8) || tc_mbar_wait(&full[i], 1, 1000);
    tc_mbar_wait(&adone[0], 0, kTcTimeoutNs / 8);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tbase, ncols);
  if (!ok || a.nsplit == 1) return;
  if (tc_last_of_tile(a.cnt + (size_t)blockIdx.y * gridDim.x / a.nsplit + tile, a.nsplit)) {
    // the tile's last CTA: partial sums in split order (then silu(gate) * up);
    // four consecutive rows per thread, every split's loads in flight at once
    const int per = NA == 2 ? 2 : 1;
    for (int i = tid; i < (kTcM / 4) * bt.ntok; i += kTcThreads) {
      const int n = i / (kTcM / 4), row = m0 + 4 * (i - n * (kTcM / 4));
      if (row >= a.rows) continue;  // rows is a multiple of 64
      const float4* pp = reinterpret_cast<const float4*>(a.part + ((size_t)bt.first + n) * per * a.rows + row);
      const size_t qs = pc * per * a.rows / 4, us = a.rows / 4;
      float4 gq[kTcMaxSplit], uq[kTcMaxSplit];
#pragma unroll
      for (int q = 0; q < kTcMaxSplit; ++q)
        if (q < a.nsplit) {
          gq[q] = __ldcg(pp + q * qs);
          if (NA == 2) uq[q] = __ldcg(pp + q * qs + us);
        }
      float4 g = gq[0], u = NA == 2 ? uq[0] : gq[0];
#pragma unroll
      for (int q = 1; q < kTcMaxSplit; ++q)
        if (q < a.nsplit) {
          g.x += gq[q].x; g.y += gq[q].y; g.z += gq[q].z; g.w += gq[q].w;
          if (NA == 2) {
            u.x += uq[q].x; u.y += uq[q].y; u.z += uq[q].z; u.w += uq[q].w;
          }
        }
      float4 h = g;
      if (NA == 2) {
        h.x = g.x / (1.f + expf(-g.x)) * u.x;
        h.y = g.y / (1.f + expf(-g.y)) * u.y;
        h.z = g.z / (1.f + expf(-g.z)) * u.z;
        h.w = g.w / (1.f + expf(-g.w)) * u.w;
      }
      *reinterpret_cast<float4*>(a.out + ((size_t)ptok[n] * a.nslot + pslot[n]) * a.rows + row) = h;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int tc_npad_max(int B) {
  const int n = B < 256 ? B : 256;
  return (n + 15) & ~15;
}

// K splits: about eight 64-column steps per CTA for gate/up (d columns), four
// for down (f columns), at most eight splits.
static int tc_split_gu(int d) {
  const int n = d / kTcBK / 8;
  return n < 1 ? 1 : (n > kTcMaxSplit ? kTcMaxSplit : n);
}
static int tc_split_dn(int f) {
  const int n = f / kTcBK / 4;
  return n < 1 ? 1 : (n > kTcMaxSplit ? kTcMaxSplit : n);
}
static size_t tc_up256(size_t n) { return (n + 255) & ~(size_t)255; }

size_t tc_split_part_bytes(int d, int f, int B, int K) {
  const size_t pc = (size_t)plan_max_pairs(B, K);
  const size_t pg = (size_t)tc_split_gu(d) * pc * 2 * f, pd = (size_t)tc_split_dn(f) * pc * d;
  return tc_up256((pg > pd ? pg : pd) * 4);
}
constexpr int kTcCntBatch = 256;  // the largest batch of any call
size_t tc_split_cnt_bytes(int d, int f, int K) {
  const size_t tiles = (size_t)((d > f ? d : f) + kTcM - 1) / kTcM;
  return tc_up256(tiles * plan_max_big(kTcCntBatch, K) * 4);
}
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
// apart), in boxes of box_bytes x 128 rows x 1 expert.
static bool make_map(CUtensorMap* m, const void* base, int row_bytes, int rows, int nexp, long long estride,
                     int box_bytes) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc || !base || (uintptr_t)base % 16 || row_bytes % 16 || estride % 16 || box_bytes % 16) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)rows, (cuuint64_t)nexp};
  const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)estride};
  const cuuint32_t box[3] = {(cuuint32_t)box_bytes, (cuuint32_t)kTcM, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the gate/up (gu) or down matrices of the routed pool and the
// shared expert. y0 receives each matrix's first row in its map's expert region.
static bool tc_maps(const ExpertSet& es, bool gu, TcMaps& M, int (&y0)[2][2]) {
  const int d = es.d, f = es.f, bits = es.bits;
  const int kc = gu ? d : f, rows = gu ? f : d;
  const int rb = kc * bits / 8, sbb = (kc / kGroup) * 4, qb = kTcBK * bits / 8;
  const long long mw = (long long)d * f * bits / 32, mg = (long long)d * f / kGroup * 2;
  memset(&M, 0, sizeof(M));
  // the shared expert (or the one explicit expert): each matrix its own view
  const void* sq[2] = {gu ? (const void*)es.shared.gate_q : (const void*)es.shared.down_q,
                       (const void*)es.shared.up_q};
  const void* ss[2] = {gu ? (const void*)es.shared.gate_sb : (const void*)es.shared.down_sb,
                       (const void*)es.shared.up_sb};
  for (int i = 0; i < (gu ? 2 : 1); ++i) {
    if (!make_map(&M.q[1][i], sq[i], rb, rows, 1, (long long)rb * rows, qb)) return false;
    if (!make_map(&M.sb[1][i], ss[i], sbb, rows, 1, (long long)sbb * rows, 16)) return false;
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
  if (!make_map(&M.q[0][0], pq, rb, region, nexp, es.q_stride * 4, qb)) return false;
  if (!make_map(&M.sb[0][0], ps, sbb, region, nexp, es.sb_stride * 2, 16)) return false;
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
  return encode_tiled() != nullptr && tc_maps(es, true, M, y0) && tc_maps(es, false, M, y0);
}

template <int BITS>
static cudaError_t tc_run(const ExpertSet& es, bool gu, const Plan* plan, int B, int K, const void* src, float* out,
                          int nslot, Ctrl* ctrl, const TcSplit& sp, cudaStream_t s) {
  TcMaps M;
  TcArgs a{};
  if (!tc_maps(es, gu, M, a.y0)) return cudaErrorInvalidValue;
  const int nbig_max = plan_max_big(B, K);
  const int npad = tc_npad_max(B);
  a.plan = plan;
  a.B = B;
  a.K = K;
  a.rows = gu ? es.f : es.d;
  a.kcols = gu ? es.d : es.f;
  a.nsplit = gu ? tc_split_gu(es.d) : tc_split_dn(es.f);
  a.rtot = tc_act_rows(B, K);
  a.act = sp.act;
  a.act_sh = reinterpret_cast<const int*>(sp.act + tc_up256((size_t)a.rtot * (((es.d > es.f ? es.d : es.f)) / kTcBK) * 128));
  a.out = out;
  a.nslot = nslot;
  a.ctrl = ctrl;
  a.part = sp.part;
  a.cnt = sp.cnt;
  int* act_sh = const_cast<int*>(a.act_sh);
  // stage the activations once
  dim3 ga(nbig_max, (npad + 7) / 8);
  if (gu)
    k_tc_act<BITS, false><<<ga, 256, 0, s>>>(plan, B, K, src, nslot, a.kcols, sp.act, act_sh, a.rtot);
  else
    k_tc_act<BITS, true><<<ga, 256, 0, s>>>(plan, B, K, src, nslot, a.kcols, sp.act, act_sh, a.rtot);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t sm = tc_gemm_smem(gu ? 2 : 1, BITS, npad);
  void* kern = gu ? (void*)k_tc_gemm<BITS, 2> : (void*)k_tc_gemm<BITS, 1>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid((a.rows + kTcM - 1) / kTcM * a.nsplit, nbig_max);
  if (gu)
    k_tc_gemm<BITS, 2><<<grid, kTcThreads, sm, s>>>(M, a);
  else
    k_tc_gemm<BITS, 1><<<grid, kTcThreads, sm, s>>>(M, a);
  return cudaGetLastError();
}

cudaError_t launch_gateup_tc(const ExpertSet& es, const Plan* plan, int B, int K, const uint16_t* x, float* H,
                             int nslot, Ctrl* ctrl, const TcSplit& sp, cudaStream_t s) {
  if (B < kBigTok) return cudaSuccess;  // no task can have 16 tokens
  return es.bits == 4 ? tc_run<4>(es, true, plan, B, K, x, H, nslot, ctrl, sp, s)
                      : tc_run<2>(es, true, plan, B, K, x, H, nslot, ctrl, sp, s);
}

cudaError_t launch_down_tc(const ExpertSet& es, const Plan* plan, int B, int K, const float* H, float* Y, int nslot,
                           Ctrl* ctrl, const TcSplit& sp, cudaStream_t s) {
  if (B < kBigTok) return cudaSuccess;
  return es.bits == 4 ? tc_run<4>(es, false, plan, B, K, H, Y, nslot, ctrl, sp, s)
                      : tc_run<2>(es, false, plan, B, K, H, Y, nslot, ctrl, sp, s);
}

}  // namespace bgq
