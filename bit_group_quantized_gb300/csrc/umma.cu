// umma.cu — tensor-core (tcgen05) grouped GEMM for experts with many tokens.
//
// When a batch routes enough tokens to one expert (16 for an explicit expert,
// 64 in a layer call, where the grouped GEMVs measured faster below that;
// always true for the shared expert at batch >= 64), the expert's three
// matrices are a dense
// contraction: rows x K weights against K x tokens activations. Here the
// weights are dequantised (w = q*scale + bias, Flash-MoE page, "FMA Dequant")
// to fp16 in shared memory, the tokens' inputs are converted to fp16 next to
// them, and tcgen05.mma (kind::f16, fp32 accumulation in tensor memory)
// multiplies them. fp16 keeps 11 significant bits, so each dequantised weight
// carries one fp16 rounding (about 2^-12 relative), far inside the layer's
// tolerance; the accumulation is fp32.
//
// Tile: 128 weight rows (M) x Npad tokens (N = the task's tokens rounded up
// to 16), K in steps of 64 (one quantisation group). Two shared-memory stages:
// while the tensor core multiplies one stage, 256 threads (two per weight row)
// fill the other; raw codes, scale/bias and activations of the next K steps
// are in flight in a cp.async ring meanwhile.
// Operands use the canonical no-swizzle K-major layout: 8x16-byte core
// matrices, the next core matrix along K 128 bytes on (LBO), the next 8 rows
// 1024 bytes on (SBO). Within each 16-column block the columns are stored in
// the order the code extraction produces them; activations use the same order,
// so every dot product is unchanged.
//
// One thread issues the MMAs and commits them to a per-stage mbarrier; every
// wait is bounded (on expiry: BGQ_ERR_TIMEOUT in the status word, a second
// bounded wait for the tensor core, tensor memory freed, return).
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

// Shared memory of one CTA: [mbar x2][tmem slot] then two stages of
// NA weight tiles (16 KB each) and one activation tile (Npad*128 bytes), then
// the rings of data in flight for D K steps: per step and row NA code slices
// (qb bytes each), per step, row and half NA scale/bias words, per step the task's
// raw activations (Npad x 4 items of 16 values, ab bytes per item).
struct TcSmem {
  uint64_t* mbar;
  uint32_t* tslot;
  unsigned char* stage[2];
  unsigned char* ringq;
  uint32_t* rings;
  unsigned char* ringa;
  int a_bytes, b_off;
};
__host__ __device__ inline size_t tc_ring_bytes(int na, int bits, int npad, int ab, int D) {
  return (size_t)D * ((size_t)kTcM * na * (kTcBK * bits / 8 + 2 * 4) + (size_t)npad * 4 * ab);
}
__device__ __forceinline__ TcSmem tc_carve(unsigned char* smem, int na, int npad, int bits, int D) {
  TcSmem S;
  S.mbar = reinterpret_cast<uint64_t*>(smem);
  S.tslot = reinterpret_cast<uint32_t*>(smem + 16);
  S.a_bytes = kTcM * kTcBK * 2;  // 16 KB
  S.b_off = na * S.a_bytes;
  const int stage_bytes = S.b_off + npad * kTcBK * 2;
  S.stage[0] = smem + 1024;
  S.stage[1] = smem + 1024 + stage_bytes;
  S.ringq = smem + 1024 + 2 * stage_bytes;
  S.rings = reinterpret_cast<uint32_t*>(S.ringq + (size_t)D * kTcM * na * (kTcBK * bits / 8));
  S.ringa = reinterpret_cast<unsigned char*>(S.rings + (size_t)D * kTcM * na * 2);
  return S;
}
size_t tc_smem_bytes(int na, int npad, int bits, int ab, int D) {
  return 1024 + 2 * ((size_t)na * kTcM * kTcBK * 2 + (size_t)npad * kTcBK * 2) + tc_ring_bytes(na, bits, npad, ab, D);
}

__device__ __forceinline__ void tc_fail(Ctrl* ctrl) { atomicExch(&ctrl->status, BGQ_ERR_TIMEOUT); }

constexpr int kTcMaxSplit = 8;  // K splits per tile (partial sums reduced by the tile's last CTA)

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
// gate/up + SiLU*mul: blockIdx.x = tile of 128 rows of d_ff x nsplit K ranges,
// blockIdx.y = big task.
// ---------------------------------------------------------------------------
template <int BITS, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
k_gateup_tc(ExpertSet es, const Plan* __restrict__ plan, int B, int K, const uint16_t* __restrict__ x,
            float* __restrict__ H, int nslot, Ctrl* ctrl, TcSplit sp, int nsplit) {
  extern __shared__ __align__(1024) unsigned char smem[];
  if ((int)blockIdx.y >= plan->nbig) return;
  const BigTask bt = plan_big(plan, B, K)[blockIdx.y];
  const int* ptok = plan_ptok(plan, B, K) + bt.first;
  const int* pslot = plan_pslot(plan, B, K) + bt.first;
  const int d = es.d, f = es.f;
  const int npad = (bt.ntok + 15) & ~15;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int tile = blockIdx.x / nsplit, split = blockIdx.x - tile * nsplit;
  const int m0 = tile * kTcM;
  TcSmem S = tc_carve(smem, 2, npad, BITS, D);
  const ExpertRef ex = tc_resolve(es, bt.expert);
  const int wpr = d * BITS / 32, gpr = d / kGroup;
  uint32_t ncols = 32;
  while ((int)ncols < 2 * npad) ncols <<= 1;
  constexpr int qb = kTcBK * BITS / 8;  // code bytes of one row and K step
  constexpr int ab = 32;                // bytes of one activation item (16 bf16)
  const int rr = tid & (kTcM - 1), hf = tid >> 7;  // tile row and half K step of this thread
  const int rme = m0 + rr;                          // the row this thread copies and dequantises
  // Step kb into ring slot kb % D: raw codes (this thread's half) and scale/bias of row rme (gate
  // and up) and this thread's activation items; one commit group per step.
  auto issue = [&](int kb, int nk_) {
    if (kb < nk_) {
      const int slot = kb % D;
      for (int i = tid; i < npad * 4; i += kTcThreads) {
        const int n = i >> 2, blk = i & 3;
        if (n < bt.ntok) {
          const uint16_t* src = x + (size_t)ptok[n] * d + kb * kTcBK + blk * 16;
          unsigned char* dst = S.ringa + ((size_t)slot * npad * 4 + i) * ab;
          cp_async16(dst, src);
          cp_async16(dst + 16, src + 8);
        }
      }
    }
    if (kb < nk_ && rme < f) {
      const int slot = kb % D;
      unsigned char* dq = S.ringq + ((size_t)(slot * kTcM + rr) * 2) * qb + hf * (qb / 2);
      const uint32_t* g = ex.gate_q + (size_t)rme * wpr + kb * (kTcBK * BITS / 32) + hf * (qb / 8);
      const uint32_t* u = ex.up_q + (size_t)rme * wpr + kb * (kTcBK * BITS / 32) + hf * (qb / 8);
      if (qb / 2 == 16) {
        cp_async16(dq, g);
        cp_async16(dq + qb, u);
      } else {
        cp_async8(dq, g);
        cp_async8(dq + qb, u);
      }
      uint32_t* ds = S.rings + ((slot * kTcM + rr) * 2 + hf) * 2;  // each half keeps its own copy
      cp_async4(ds, reinterpret_cast<const uint32_t*>(ex.gate_sb) + (size_t)rme * gpr + kb);
      cp_async4(ds + 1, reinterpret_cast<const uint32_t*>(ex.up_sb) + (size_t)rme * gpr + kb);
    }
    cp_async_commit();
  };

  if (tid == 0) {
    tc_mbar_init(&S.mbar[0]);
    tc_mbar_init(&S.mbar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(S.tslot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *S.tslot;
  const uint32_t idesc = tc_idesc(npad);
  const int nkt = d / kTcBK;  // K steps of the whole row; this CTA takes [kb0, nk)
  const int kb0 = nkt * split / nsplit, nk = nkt * (split + 1) / nsplit;
  bool ok = true;
  for (int kb = kb0; kb < kb0 + D - 1; ++kb) issue(kb, nk);

  for (int kb = kb0; kb < nk; ++kb) {
    const int j = kb - kb0;  // local step: stage and mbarrier phase
    const int s = j & 1;
    unsigned char* st = S.stage[s];
    issue(kb + D - 1, nk);
    cp_async_wait<D - 1>();  // this thread's copies of step kb have landed
    if (j >= 2 && !tc_mbar_wait(&S.mbar[s], (uint32_t)((j / 2 - 1) & 1), kTcTimeoutNs)) {
      ok = false;
      break;
    }
    // weights: this thread dequantises its half of row rme of gate and of up
    {
      if (rme < f) {
        const int slot = kb % D;
        const unsigned char* dq = S.ringq + ((size_t)(slot * kTcM + rr) * 2) * qb + hf * (qb / 2);
        const uint32_t* ds = S.rings + ((slot * kTcM + rr) * 2 + hf) * 2;
        dequant_half<BITS>(reinterpret_cast<const uint32_t*>(dq), ds[0], st, rr, hf);
        dequant_half<BITS>(reinterpret_cast<const uint32_t*>(dq + qb), ds[1], st + S.a_bytes, rr, hf);
      } else {
#pragma unroll
        for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
          *reinterpret_cast<uint4*>(st + tc_off(rr, c >> 1, (c & 1) * 8)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(st + S.a_bytes + tc_off(rr, c >> 1, (c & 1) * 8)) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    // activations: (token n, 16-column block) per thread, from the ring
    for (int i = tid; i < npad * 4; i += kTcThreads) {
      const int n = i >> 2, blk = i & 3;
      float v[16];
      if (n < bt.ntok) {
        const unsigned char* xp = S.ringa + ((size_t)(kb % D) * npad * 4 + i) * ab;
        unpack_bf16x8(*reinterpret_cast<const uint4*>(xp), v);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(xp + 16), v + 8);
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = 0.f;
      }
      put_act16<BITS>(st + S.b_off, n, blk, v);
    }
    tc_fence_proxy();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int jj = 0; jj < kTcBK / 16; ++jj) {
        const uint64_t bd = tc_desc(st + S.b_off + jj * 256);
        tc_mma(tbase, tc_desc(st + jj * 256), bd, idesc, (j | jj) ? 1u : 0u);
        tc_mma(tbase + npad, tc_desc(st + S.a_bytes + jj * 256), bd, idesc, (j | jj) ? 1u : 0u);
      }
      tc_commit(&S.mbar[s]);
    }
  }
  cp_async_wait_all();
  // the last commit covers every MMA
  const int nl = nk - kb0;
  if (ok) ok = tc_mbar_wait(&S.mbar[(nl - 1) & 1], (uint32_t)(((nl - 1) / 2) & 1), kTcTimeoutNs);
  const size_t pc = (size_t)plan_max_pairs(B, K);
  if (ok && warp < 4) {  // warp w reads tensor-memory lanes 32w..32w+31
    tc_fence_after();
    const int row = m0 + warp * 32 + (tid & 31);
    for (int c0 = 0; c0 < npad; c0 += 8) {
      float g[8], u[8];
      const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
      tmem_ld8(tbase + lane_off + c0, g);
      tmem_ld8(tbase + lane_off + npad + c0, u);
      if (row < f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + i;
          if (n >= bt.ntok) continue;
          if (nsplit == 1) {
            H[((size_t)ptok[n] * nslot + pslot[n]) * f + row] = g[i] / (1.f + expf(-g[i])) * u[i];
          } else {  // partial sums of this K range: [split][pair][gate, up][row]
            float* pp = sp.part + (((size_t)split * pc + bt.first + n) * 2) * f + row;
            pp[0] = g[i];
            pp[f] = u[i];
          }
        }
      }
    }
  } else if (!ok) {
    if (tid == 0) tc_fail(ctrl);
    // give the tensor core a last bounded chance to finish before the memory is freed
    tc_mbar_wait(&S.mbar[0], 0, kTcTimeoutNs / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tbase, ncols);
  if (nsplit > 1 && tc_last_of_tile(sp.cnt + (size_t)blockIdx.y * gridDim.x / nsplit + tile, nsplit)) {
    // the tile's last CTA: partial sums in split order, then SiLU(gate) * up;
    // four consecutive rows per thread, every split's loads in flight at once
    for (int i = tid; i < (kTcM / 4) * bt.ntok; i += kTcThreads) {
      const int n = i / (kTcM / 4), row = m0 + 4 * (i - n * (kTcM / 4));
      if (row >= f) continue;  // f is a multiple of 64
      const float4* pp = reinterpret_cast<const float4*>(sp.part + ((size_t)bt.first + n) * 2 * f + row);
      const size_t qs = pc * 2 * f / 4, us = f / 4;
      float4 gq[kTcMaxSplit], uq[kTcMaxSplit];
#pragma unroll
      for (int q = 0; q < kTcMaxSplit; ++q)
        if (q < nsplit) {
          gq[q] = __ldcg(pp + q * qs);
          uq[q] = __ldcg(pp + q * qs + us);
        }
      float4 g = gq[0], u = uq[0];
#pragma unroll
      for (int q = 1; q < kTcMaxSplit; ++q)
        if (q < nsplit) {
          g.x += gq[q].x; g.y += gq[q].y; g.z += gq[q].z; g.w += gq[q].w;
          u.x += uq[q].x; u.y += uq[q].y; u.z += uq[q].z; u.w += uq[q].w;
        }
      float4 h;
      h.x = g.x / (1.f + expf(-g.x)) * u.x;
      h.y = g.y / (1.f + expf(-g.y)) * u.y;
      h.z = g.z / (1.f + expf(-g.z)) * u.z;
      h.w = g.w / (1.f + expf(-g.w)) * u.w;
      *reinterpret_cast<float4*>(H + ((size_t)ptok[n] * nslot + pslot[n]) * f + row) = h;
    }
  }
}

// ---------------------------------------------------------------------------
// down projection: blockIdx.x = tile of 128 rows of d_model x nsplit K ranges,
// blockIdx.y = big task.
// ---------------------------------------------------------------------------
template <int BITS, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
k_down_tc(ExpertSet es, const Plan* __restrict__ plan, int B, int K, const float* __restrict__ H,
          float* __restrict__ Y, int nslot, Ctrl* ctrl, TcSplit sp, int nsplit) {
  extern __shared__ __align__(1024) unsigned char smem[];
  if ((int)blockIdx.y >= plan->nbig) return;
  const BigTask bt = plan_big(plan, B, K)[blockIdx.y];
  const int* ptok = plan_ptok(plan, B, K) + bt.first;
  const int* pslot = plan_pslot(plan, B, K) + bt.first;
  const int d = es.d, f = es.f;
  const int npad = (bt.ntok + 15) & ~15;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int tile = blockIdx.x / nsplit, split = blockIdx.x - tile * nsplit;
  const int m0 = tile * kTcM;
  TcSmem S = tc_carve(smem, 1, npad, BITS, D);
  const ExpertRef ex = tc_resolve(es, bt.expert);
  const int wpr = f * BITS / 32, gpr = f / kGroup;
  uint32_t ncols = 32;
  while ((int)ncols < npad) ncols <<= 1;
  constexpr int qb = kTcBK * BITS / 8;
  constexpr int ab = 64;  // bytes of one activation item (16 fp32)
  const int rr = tid & (kTcM - 1), hf = tid >> 7;  // tile row and half K step of this thread
  const int rme = m0 + rr;
  auto issue = [&](int kb, int nk_) {
    if (kb < nk_) {
      const int slot = kb % D;
      for (int i = tid; i < npad * 4; i += kTcThreads) {
        const int n = i >> 2, blk = i & 3;
        if (n < bt.ntok) {
          const float* src = H + ((size_t)ptok[n] * nslot + pslot[n]) * f + kb * kTcBK + blk * 16;
          unsigned char* dst = S.ringa + ((size_t)slot * npad * 4 + i) * ab;
#pragma unroll
          for (int o = 0; o < 4; ++o) cp_async16(dst + 16 * o, src + 4 * o);
        }
      }
    }
    if (kb < nk_ && rme < d) {
      const int slot = kb % D;
      unsigned char* dq = S.ringq + (size_t)(slot * kTcM + rr) * qb + hf * (qb / 2);
      const uint32_t* q = ex.down_q + (size_t)rme * wpr + kb * (kTcBK * BITS / 32) + hf * (qb / 8);
      if (qb / 2 == 16)
        cp_async16(dq, q);
      else
        cp_async8(dq, q);
      cp_async4(S.rings + (slot * kTcM + rr) * 2 + hf,
                reinterpret_cast<const uint32_t*>(ex.down_sb) + (size_t)rme * gpr + kb);
    }
    cp_async_commit();
  };

  if (tid == 0) {
    tc_mbar_init(&S.mbar[0]);
    tc_mbar_init(&S.mbar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(S.tslot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *S.tslot;
  const uint32_t idesc = tc_idesc(npad);
  const int nkt = f / kTcBK;  // K steps of the whole row; this CTA takes [kb0, nk)
  const int kb0 = nkt * split / nsplit, nk = nkt * (split + 1) / nsplit;
  bool ok = true;
  for (int kb = kb0; kb < kb0 + D - 1; ++kb) issue(kb, nk);

  for (int kb = kb0; kb < nk; ++kb) {
    const int j = kb - kb0;  // local step: stage and mbarrier phase
    const int s = j & 1;
    unsigned char* st = S.stage[s];
    issue(kb + D - 1, nk);
    cp_async_wait<D - 1>();
    if (j >= 2 && !tc_mbar_wait(&S.mbar[s], (uint32_t)((j / 2 - 1) & 1), kTcTimeoutNs)) {
      ok = false;
      break;
    }
    {
      if (rme < d) {
        const int slot = kb % D;
        dequant_half<BITS>(
            reinterpret_cast<const uint32_t*>(S.ringq + (size_t)(slot * kTcM + rr) * qb + hf * (qb / 2)),
            S.rings[(slot * kTcM + rr) * 2 + hf], st, rr, hf);
      } else {
#pragma unroll
        for (int c = 4 * hf; c < 4 * hf + 4; ++c)
          *reinterpret_cast<uint4*>(st + tc_off(rr, c >> 1, (c & 1) * 8)) = make_uint4(0, 0, 0, 0);
      }
    }
    for (int i = tid; i < npad * 4; i += kTcThreads) {
      const int n = i >> 2, blk = i & 3;
      float v[16];
      if (n < bt.ntok) {
        const float* hp = reinterpret_cast<const float*>(S.ringa + ((size_t)(kb % D) * npad * 4 + i) * ab);
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
          const float4 a = *reinterpret_cast<const float4*>(hp + k);
          v[k] = a.x;
          v[k + 1] = a.y;
          v[k + 2] = a.z;
          v[k + 3] = a.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = 0.f;
      }
      put_act16<BITS>(st + S.b_off, n, blk, v);
    }
    tc_fence_proxy();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int jj = 0; jj < kTcBK / 16; ++jj)
        tc_mma(tbase, tc_desc(st + jj * 256), tc_desc(st + S.b_off + jj * 256), idesc, (j | jj) ? 1u : 0u);
      tc_commit(&S.mbar[s]);
    }
  }
  cp_async_wait_all();
  const int nl = nk - kb0;
  if (ok) ok = tc_mbar_wait(&S.mbar[(nl - 1) & 1], (uint32_t)(((nl - 1) / 2) & 1), kTcTimeoutNs);
  const size_t pc = (size_t)plan_max_pairs(B, K);
  if (ok && warp < 4) {  // warp w reads tensor-memory lanes 32w..32w+31
    tc_fence_after();
    const int row = m0 + warp * 32 + (tid & 31);
    for (int c0 = 0; c0 < npad; c0 += 8) {
      float y[8];
      tmem_ld8(tbase + ((uint32_t)(warp * 32) << 16) + c0, y);
      if (row < d) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + i;
          if (n >= bt.ntok) continue;
          if (nsplit == 1)
            Y[((size_t)ptok[n] * nslot + pslot[n]) * d + row] = y[i];
          else  // partial sums of this K range: [split][pair][row]
            sp.part[((size_t)split * pc + bt.first + n) * d + row] = y[i];
        }
      }
    }
  } else if (!ok) {
    if (tid == 0) tc_fail(ctrl);
    tc_mbar_wait(&S.mbar[0], 0, kTcTimeoutNs / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tbase, ncols);
  if (nsplit > 1 && tc_last_of_tile(sp.cnt + (size_t)blockIdx.y * gridDim.x / nsplit + tile, nsplit)) {
    for (int i = tid; i < (kTcM / 4) * bt.ntok; i += kTcThreads) {
      const int n = i / (kTcM / 4), row = m0 + 4 * (i - n * (kTcM / 4));
      if (row >= d) continue;  // d is a multiple of 64
      const float4* pp = reinterpret_cast<const float4*>(sp.part + ((size_t)bt.first + n) * d + row);
      const size_t qs = pc * d / 4;
      float4 yq[kTcMaxSplit];
#pragma unroll
      for (int q = 0; q < kTcMaxSplit; ++q)
        if (q < nsplit) yq[q] = __ldcg(pp + q * qs);
      float4 y = yq[0];
#pragma unroll
      for (int q = 1; q < kTcMaxSplit; ++q)
        if (q < nsplit) {
          y.x += yq[q].x; y.y += yq[q].y; y.z += yq[q].z; y.w += yq[q].w;
        }
      *reinterpret_cast<float4*>(Y + ((size_t)ptok[n] * nslot + pslot[n]) * d + row) = y;
    }
  }
}

// ---------------------------------------------------------------------------
static int tc_npad_max(int B) {
  int n = B < 256 ? B : 256;
  return (n + 15) & ~15;
}

// Ring depth by the task width (shared memory: the rings grow with Npad).
static int tc_depth(int npad, bool down) {
  if (npad <= 64) return 8;
  if (npad <= 128) return 4;
  return down ? 1 : 2;
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

template <int BITS, int D>
static cudaError_t gateup_tc_d(const ExpertSet& es, const Plan* plan, int B, int K, const uint16_t* x, float* H,
                               int nslot, Ctrl* ctrl, const TcSplit& sp, int npad, cudaStream_t s) {
  const size_t sm = tc_smem_bytes(2, npad, BITS, 32, D);
  cudaError_t e = cudaFuncSetAttribute(k_gateup_tc<BITS, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int ns = sp.part ? tc_split_gu(es.d) : 1;
  dim3 grid((es.f + kTcM - 1) / kTcM * ns, plan_max_big(B, K));
  k_gateup_tc<BITS, D><<<grid, kTcThreads, sm, s>>>(es, plan, B, K, x, H, nslot, ctrl, sp, ns);
  return cudaGetLastError();
}
template <int BITS, int D>
static cudaError_t down_tc_d(const ExpertSet& es, const Plan* plan, int B, int K, const float* H, float* Y,
                             int nslot, Ctrl* ctrl, const TcSplit& sp, int npad, cudaStream_t s) {
  const size_t sm = tc_smem_bytes(1, npad, BITS, 64, D);
  cudaError_t e = cudaFuncSetAttribute(k_down_tc<BITS, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int ns = sp.part ? tc_split_dn(es.f) : 1;
  dim3 grid((es.d + kTcM - 1) / kTcM * ns, plan_max_big(B, K));
  k_down_tc<BITS, D><<<grid, kTcThreads, sm, s>>>(es, plan, B, K, H, Y, nslot, ctrl, sp, ns);
  return cudaGetLastError();
}

cudaError_t launch_gateup_tc(const ExpertSet& es, const Plan* plan, int B, int K, const uint16_t* x, float* H,
                             int nslot, Ctrl* ctrl, const TcSplit& sp, cudaStream_t s) {
  if (B < kBigTok) return cudaSuccess;  // no task can have 16 tokens
  const int npad = tc_npad_max(B);
  const int D = tc_depth(npad, false);
  if (es.bits == 4)
    return D == 8 ? gateup_tc_d<4, 8>(es, plan, B, K, x, H, nslot, ctrl, sp, npad, s)
                  : D == 4 ? gateup_tc_d<4, 4>(es, plan, B, K, x, H, nslot, ctrl, sp, npad, s)
                           : gateup_tc_d<4, 2>(es, plan, B, K, x, H, nslot, ctrl, sp, npad, s);
  return D == 8 ? gateup_tc_d<2, 8>(es, plan, B, K, x, H, nslot, ctrl, sp, npad, s)
                : D == 4 ? gateup_tc_d<2, 4>(es, plan, B, K, x, H, nslot, ctrl, sp, npad, s)
                         : gateup_tc_d<2, 2>(es, plan, B, K, x, H, nslot, ctrl, sp, npad, s);
}

cudaError_t launch_down_tc(const ExpertSet& es, const Plan* plan, int B, int K, const float* H, float* Y, int nslot,
                           Ctrl* ctrl, const TcSplit& sp, cudaStream_t s) {
  if (B < kBigTok) return cudaSuccess;
  const int npad = tc_npad_max(B);
  const int D = tc_depth(npad, true);
  if (es.bits == 4)
    return D == 8 ? down_tc_d<4, 8>(es, plan, B, K, H, Y, nslot, ctrl, sp, npad, s)
                  : D == 4 ? down_tc_d<4, 4>(es, plan, B, K, H, Y, nslot, ctrl, sp, npad, s)
                           : down_tc_d<4, 1>(es, plan, B, K, H, Y, nslot, ctrl, sp, npad, s);
  return D == 8 ? down_tc_d<2, 8>(es, plan, B, K, H, Y, nslot, ctrl, sp, npad, s)
                : D == 4 ? down_tc_d<2, 4>(es, plan, B, K, H, Y, nslot, ctrl, sp, npad, s)
                         : down_tc_d<2, 1>(es, plan, B, K, H, Y, nslot, ctrl, sp, npad, s);
}

}  // namespace bgq
