// fused.cu — one persistent kernel for batch-1 decode: a whole token through
// one MoE layer or a stack of layers per launch.
//
// Flash-MoE page, section "架构设计：SSD当显存用": per token and layer the path
// is routing logits -> softmax + top-K -> the selected experts' forward pass
// -> combine (-> norm). At batch 1 every step is a matrix-vector product whose
// weights are read exactly once, so a layer is bound by HBM bandwidth and by
// the latency of its three dependent steps. One cooperative launch with one
// CTA per SM keeps the token on chip and replaces kernel boundaries by
// grid-wide exchanges:
//
//   A  RMSNorm of the residual (stack mode), router rows (bf16) and the shared
//      expert's gate/up rows; every CTA publishes its logits as tagged words;
//   B  once every logit carries the layer's tag, every CTA selects the same
//      top-K experts from all logits and computes its share of their gate/up
//      rows;
//   C  after the SwiGLU counter, every CTA computes its output rows: the down
//      rows of the K selected experts and of the shared expert, combined in a
//      fixed order, plus the residual add in stack mode (after the residual
//      counter of the previous layer).
//
// Data movement. Each CTA owns a fixed slice of every phase. Its router rows,
// shared gate/up rows (phase A), selected-expert gate/up rows (phase B) and
// down rows (phase C) are streamed into shared memory with bulk async copies
// (cp.async.bulk, one mbarrier per work unit), each issued as soon as it is
// known and its buffer is free: phase B's right after the selection, phase C's
// right after phase B (they land while the grid waits at the SwiGLU counter),
// the next layer's phase A's once that wait is over (issued before it, they
// slowed the exchange: 21.3 vs 21.0 us per layer). Consumers start on a unit
// as soon as its own mbarrier completes.
//
// Exchanges. The logits (2 KB) go as 64-bit {value, layer + 1} words written
// with relaxed stores and polled by every thread for its share: a reader that
// sees the tag sees the value, so no fence and no counter are needed (20.74 ->
// 19.98 us per layer against a counter barrier plus a separate read; the
// words are zero at every launch's start, the last CTA out clears them). The
// SwiGLU outputs (20 KB per CTA) and the residual use counters: a CTA's
// release reduction after a block barrier, thread 0 polling with acquire
// loads. (Tagged words for the SwiGLU outputs measured 24.90 against 20.01 us
// per layer: their polls slowed the last CTAs' phase-B copies; an earlier
// variant with all three exchanges tagged, 29.5 against 24.8 us.)
//
// Every wait is bounded (an iteration count and %globaltimer). On expiry the
// CTA sets BGQ_ERR_TIMEOUT in the status word and an abort flag that makes
// every CTA leave at its next grid-wide wait; before leaving, thread 0 waits
// (again with a limit) for the bulk copies its CTA still has in flight.
#include <climits>

#include "../../include/bgq.h"
#include "common.cuh"
#include "fused.h"
#include "topk.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kMaxS1 = 16;   // shared gate/up units per CTA
constexpr int kMaxB = 32;    // selected gate/up units per CTA
constexpr int kCH = 14;      // units per bulk-copy chunk (one mbarrier per chunk)
constexpr int kMaxSC = 4;    // shared gate/up chunks per CTA
constexpr int kMaxBC = 16;   // selected gate/up chunks per CTA
constexpr long long kMaxSpin = 1ll << 26;
constexpr long long kDrainNs = 200000000ll;

// --------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* m, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* m, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity)
      : "memory");
  return ok != 0;
}
// global -> shared bulk copy, completion counted on mbarrier m (16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* m) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(m))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ bool aborted(Ctrl* ctrl) { return *(volatile int*)&ctrl->misc[0] != 0; }
__device__ __forceinline__ void raise_timeout(Ctrl* ctrl) {
  atomicExch(&ctrl->status, BGQ_ERR_TIMEOUT);
  atomicExch(&ctrl->misc[0], 1);
}

// Bounded wait for mbarrier phase `parity`; false on timeout or abort.
__device__ bool mbar_wait(uint64_t* m, uint32_t parity, Ctrl* ctrl, long long timeout_ns) {
  if (mbar_try_wait(m, parity)) return true;
  const unsigned long long t0 = globaltimer();
  long long it = 0;
  while (!mbar_try_wait(m, parity)) {
    if ((++it & 31) == 0) {
      if (aborted(ctrl)) return false;
      if (it > kMaxSpin || (long long)(globaltimer() - t0) > timeout_ns) {
        raise_timeout(ctrl);
        return false;
      }
    }
  }
  return true;
}

// --------------------------------------------------------------- geometry
// Row shapes handled here: rows of d (router, gate, up) are read by all 32
// lanes (d*bits/128 parts, a multiple of 32, at most 4 per lane); rows of f
// (down) have at most 32 parts, one per lane.
struct FGeo {
  int nC;          // CTAs
  int qr;          // warps per router row (1024 columns each)
  int rpc;         // router rows per CTA
  int nRouter;     // CTAs holding router rows
  int s1_nr;       // shared gate/up units per CTA without router rows
  int nit_d;       // parts per lane of a d-row
  int wpr, gpr;    // words / groups per d-row
  int unit;        // bytes of one gate+up unit in shared memory
  int nBmax;       // selected gate/up units per CTA (max)
  int bufA, bufB;  // shared-memory buffer bytes
};

__host__ __device__ inline void fsplit(int n, int part, int nparts, int& b, int& e) {
  b = (int)((long long)n * part / nparts);
  e = (int)((long long)n * (part + 1) / nparts);
}

__host__ __device__ inline FGeo fgeo(int nC, int d, int f, int E, int K, int bits) {
  FGeo g;
  g.nC = nC;
  g.qr = (d >= 1024 && d % 1024 == 0) ? d / 1024 : 1;
  g.rpc = kFWarps / g.qr;
  g.nRouter = (E + 1 + g.rpc - 1) / g.rpc;
  g.nit_d = d * bits / 128 / 32;
  g.wpr = d * bits / 32;
  g.gpr = d / kGroup;
  g.unit = 2 * (g.wpr + g.gpr) * 4;
  g.nBmax = (K * f + nC - 1) / nC;
  const int n_nr = nC - g.nRouter;
  g.s1_nr = 0;
  if (n_nr > 0) {
    // balance phase A's bytes: a router row is 2d bytes, a gate+up unit `unit` bytes
    double total = (double)(E + 1) * 2 * d + (double)f * g.unit;
    int a = (int)(total / nC / g.unit + 0.5);
    if (a * n_nr > f) a = f / n_nr;
    if (a > kMaxS1) a = kMaxS1;
    g.s1_nr = a < 0 ? 0 : a;
  }
  const int rest = f - n_nr * g.s1_nr;
  const int nparts = g.s1_nr > 0 ? g.nRouter : nC;
  const int s1_router = (rest + nparts - 1) / nparts;
  int a_router = g.rpc * 2 * d + s1_router * g.unit;
  int a_nr = g.s1_nr * g.unit;
  g.bufA = a_router > a_nr ? a_router : a_nr;
  g.bufB = g.nBmax * g.unit;
  // phase C reuses bufB for its down rows (K+1 experts x the CTA's rows) and partial results
  const int rows_c = (d + nC - 1) / nC;
  // ... followed by the SwiGLU outputs gathered as fp32, then staged
  const int c_bytes = (K + 1) * rows_c * (f * bits / 8 + (f / kGroup) * 4) + (K + 1) * rows_c * 4 + 48 +
                      (K + 1) * f * 4 + (int)xstage_bytes(K + 1, f, bits);
  if (g.bufB < c_bytes) g.bufB = c_bytes;
  // the selection's logits and scratch live in bufB before phase B's copies
  const int sel_bytes = (((E + 4) & ~3) + topk_scratch_ints(E)) * 4;
  if (g.bufB < sel_bytes) g.bufB = sel_bytes;
  return g;
}

// Shared-memory layout (byte offsets; every region 128-byte aligned).
struct FLayout {
  size_t misc, rho, a_s, sta, hres, bufA, bufB, total;
};
__host__ __device__ inline size_t fl_take(size_t& o, size_t bytes) {
  size_t r = o;
  o += (bytes + 127) & ~(size_t)127;
  return r;
}
__host__ __device__ inline FLayout flayout(const FGeo& g, int d, int f, int K, int bits) {
  FLayout L;
  size_t o = 0;
  fl_take(o, (3 + kMaxSC + kMaxBC) * 8);  // mbarriers at offset 0
  L.misc = fl_take(o, 256);
  L.rho = fl_take(o, (size_t)d * 2);  // apar, bpar, s_idx[8], s_w[9], red[kFWarps]
  L.a_s = fl_take(o, (size_t)d * 2);
  L.sta = fl_take(o, xstage_bytes(1, d, bits));  // the staged layer input (phase B's SwiGLU outputs: in bufB)
  L.hres = fl_take(o, (size_t)((d + g.nC - 1) / g.nC) * 4);  // this CTA's rows of the residual
  L.bufA = fl_take(o, (size_t)g.bufA);
  L.bufB = fl_take(o, (size_t)g.bufB);
  L.total = o;
  return L;
}

// This CTA's shared gate/up unit range.
__device__ __forceinline__ void s1_range(const FGeo& g, int f, int& b, int& e) {
  const int n_nr = g.nC - g.nRouter;
  if (g.s1_nr > 0 && (int)blockIdx.x >= g.nRouter) {
    b = ((int)blockIdx.x - g.nRouter) * g.s1_nr;
    e = b + g.s1_nr;
    return;
  }
  const int rest0 = g.s1_nr > 0 ? n_nr * g.s1_nr : 0;
  fsplit(f - rest0, blockIdx.x, g.s1_nr > 0 ? g.nRouter : g.nC, b, e);
  b += rest0;
  e += rest0;
}

// Offset of the shared gate/up units in bufA: after the router rows on CTAs
// that hold router rows, at 0 on the others (bufA is sized for both cases).
__device__ __forceinline__ size_t s1_base(const FGeo& g, int d) {
  return (int)blockIdx.x < g.nRouter ? (size_t)g.rpc * 2 * d : 0;
}

// Units [b, e) are copied in chunks of up to kCH consecutive rows that never
// cross a multiple of `seg` (an expert boundary). Chunk c holds n units laid
// out as [gate q rows][up q rows][gate sb rows][up sb rows] starting at byte
// (start - b) * unit of its buffer.
struct Chunk {
  int start, n, idx;
};
__device__ __forceinline__ Chunk chunk_at(int c, int b, int e, int seg) {
  int start = b;
  for (int i = 0; i < c && start < e; ++i) {
    int lim = min(min(start + kCH, e), (start / seg + 1) * seg);
    start = lim;
  }
  const int lim = min(min(start + kCH, e), (start / seg + 1) * seg);
  return Chunk{start, start < e ? lim - start : 0, c};
}
__device__ __forceinline__ Chunk chunk_of(int u, int b, int e, int seg) {
  int start = b, idx = 0;
  while (true) {
    const int lim = min(min(start + kCH, e), (start / seg + 1) * seg);
    if (u < lim) return Chunk{start, lim - start, idx};
    start = lim;
    ++idx;
  }
}

// --------------------------------------------------------------- compute helpers
// Gate and up rows of two units (in shared memory) against staged input 0:
// four dot products that share every x chunk load. Unit i is at position
// p_i of a chunk of n_i units starting at c_i. Lane l reads part it*32 + l.
// Returns silu(gate) * up of unit 0 in lane 0 and of unit 1 in lane 16.
template <int BITS>
__device__ __noinline__ float units_gateup2(const unsigned char* c0, int n0, int p0, const unsigned char* c1, int n1,
                                            int p1, const XStage st, const FGeo g, int lane) {
  using G = Geo<BITS>;
  const int wq = g.wpr * 4, ws = g.gpr * 4;
  const uint4* qg0 = reinterpret_cast<const uint4*>(c0 + p0 * wq);
  const uint4* qu0 = reinterpret_cast<const uint4*>(c0 + (n0 + p0) * wq);
  const uint32_t* sg0 = reinterpret_cast<const uint32_t*>(c0 + 2 * n0 * wq + p0 * ws);
  const uint32_t* su0 = reinterpret_cast<const uint32_t*>(c0 + 2 * n0 * wq + (n0 + p0) * ws);
  const uint4* qg1 = reinterpret_cast<const uint4*>(c1 + p1 * wq);
  const uint4* qu1 = reinterpret_cast<const uint4*>(c1 + (n1 + p1) * wq);
  const uint32_t* sg1 = reinterpret_cast<const uint32_t*>(c1 + 2 * n1 * wq + p1 * ws);
  const uint32_t* su1 = reinterpret_cast<const uint32_t*>(c1 + 2 * n1 * wq + (n1 + p1) * ws);
  const RowGeo rg{g.nit_d * 32, 32, 1, g.nit_d};
  float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int it = 0; it < g.nit_d; ++it) {
    const int p = it * 32 + lane, pg = part_group<BITS>(p);
    const uint4 a = qg0[p], b = qu0[p], c = qg1[p], d = qu1[p];
    const uint32_t sa = sg0[pg], sb = su0[pg], sc = sg1[pg], sd = su1[pg];
    uint4 xc[4 * G::kNch];
    uint2 xh[4 * G::kNch];
    load_part_x<BITS>(st, 0, it, lane, rg, xc, xh);
    const float2 pi = st.partinfo[p];
    v[0] = part_dot_x<BITS>(a, sa, xc, xh, pi, v[0]);
    v[1] = part_dot_x<BITS>(b, sb, xc, xh, pi, v[1]);
    v[2] = part_dot_x<BITS>(c, sc, xc, xh, pi, v[2]);
    v[3] = part_dot_x<BITS>(d, sd, xc, xh, pi, v[3]);
  }
  // lanes 0-7: gate 0, 8-15: up 0, 16-23: gate 1, 24-31: up 1 (bit-identical to warp_sum)
  const float r = row_reduce4(v, 32, lane);
  const float up = __shfl_down_sync(kFull, r, 8);
  return r / (1.f + expf(-r)) * up;
}

// Units [b, e) of a phase (chunks of kCH units that never cross a multiple of
// seg, chunk i complete on mbars[i]), two per warp: exchange word hk_dst[j] =
// silu(gate) * up of unit b + j. An odd last unit is computed twice, written once.
template <int BITS>
__device__ __forceinline__ void run_units(const unsigned char* base, int b, int e, int seg, uint64_t* mbars,
                                          uint32_t par, Ctrl* ctrl, long long timeout_ns, const XStage& st,
                                          const FGeo& g, float* hk_dst, int warp, int lane) {
  const int nu = e - b;
  for (int j0 = 2 * warp; j0 < nu; j0 += 2 * kFWarps) {
    const int j1 = min(j0 + 1, nu - 1);
    const Chunk c0 = chunk_of(b + j0, b, e, seg), c1 = chunk_of(b + j1, b, e, seg);
    mbar_wait(&mbars[c0.idx], par, ctrl, timeout_ns);
    if (c1.idx != c0.idx) mbar_wait(&mbars[c1.idx], par, ctrl, timeout_ns);
    const float h = units_gateup2<BITS>(base + (size_t)(c0.start - b) * g.unit, c0.n, b + j0 - c0.start,
                                        base + (size_t)(c1.start - b) * g.unit, c1.n, b + j1 - c1.start, st, g, lane);
    if (lane == 0) hk_dst[j0] = h;
    if (lane == 16 && j1 != j0) hk_dst[j1] = h;
  }
}

// A slice (<= 1024 columns) of a bf16 router row in shared memory dotted with
// the bf16 input in shared memory.
__device__ __forceinline__ float router_dot(const uint16_t* wrow, const uint16_t* a_s, int c0, int nvec, int lane) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < nvec) {
      const uint4 w = *reinterpret_cast<const uint4*>(wrow + c0 + (i * 32 + lane) * 8);
      const uint4 x = *reinterpret_cast<const uint4*>(a_s + c0 + (i * 32 + lane) * 8);
      acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc);
      acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
      acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc);
      acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
      acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc);
      acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
      acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc);
      acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
    }
  }
  return warp_sum(acc);
}

// x staging from fp32 values in shared memory (the layer input).
template <int BITS>
__device__ __forceinline__ void stage_f32(const float* src, int ld, int T, int cols, const XStage st) {
  stage_x24<BITS>(StridedSrc<float>{src, ld}, T, cols, st);
}
// Thread 0 stamps event ev of layer l (no-op without a trace buffer).
__device__ __forceinline__ void stamp(const FusedParams& P, int l, int ev) {
  if (P.trace && threadIdx.x == 0)
    P.trace[((size_t)l * gridDim.x + blockIdx.x) * kTraceEvents + ev] = globaltimer();
}


// Shared-memory state of the kernel.
struct FSmem {
  uint64_t* mR;    // router rows
  uint64_t* mRho;  // RMSNorm weight
  uint64_t* mC;    // down rows of phase C
  uint16_t* rho;
  uint64_t* mS;  // [kMaxSC] shared gate/up chunks
  uint64_t* mB;  // [kMaxBC] selected gate/up chunks
  unsigned char* bufA;
  unsigned char* bufB;
  int* apar;  // parity of the last issued A batch (-1: none)
  int* bpar;  // parity of the last issued B batch (-1: none)
  int* cpar;  // parity of the last issued C batch (-1: none)
};

// Thread 0: wait (bounded) for every bulk copy this CTA still has in flight.
__device__ void drain_copies(const FSmem& S) {
  const unsigned long long t0 = globaltimer();
  const int ap = *S.apar, bp = *S.bpar, cp = *S.cpar;
  if (cp >= 0)
    while (!mbar_try_wait(S.mC, (uint32_t)cp) && (long long)(globaltimer() - t0) < kDrainNs) {
    }
  if (ap >= 0) {
    while (!mbar_try_wait(S.mR, (uint32_t)ap) && (long long)(globaltimer() - t0) < kDrainNs) {
    }
    while (!mbar_try_wait(S.mRho, (uint32_t)ap) && (long long)(globaltimer() - t0) < kDrainNs) {
    }
    for (int j = 0; j < kMaxSC; ++j)
      while (!mbar_try_wait(&S.mS[j], (uint32_t)ap) && (long long)(globaltimer() - t0) < kDrainNs) {
      }
  }
  if (bp >= 0)
    for (int j = 0; j < kMaxBC; ++j)
      while (!mbar_try_wait(&S.mB[j], (uint32_t)bp) && (long long)(globaltimer() - t0) < kDrainNs) {
      }
}

// Grid-wide wait: thread 0 waits until *p >= target. False for the whole CTA
// on abort or timeout (after thread 0 drained the CTA's copies in flight).
__device__ bool cta_wait(const int* p, int target, Ctrl* ctrl, long long timeout_ns, const FSmem& S) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned long long t0 = globaltimer();
    long long it = 0;
    while (ld_acquire(p) < target) {
      if (aborted(ctrl)) {
        ok = 0;
        break;
      }
      if (++it > kMaxSpin || (long long)(globaltimer() - t0) > timeout_ns) {
        raise_timeout(ctrl);
        ok = 0;
        break;
      }
      if (it > 16) __nanosleep(32);
    }
    if (ok && aborted(ctrl)) ok = 0;
    if (!ok) drain_copies(S);
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// All threads: publish this CTA's global writes, then count it in *p
// (block barrier, then one release reduction by thread 0).
__device__ void cta_arrive(int* p) {
  __syncthreads();
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p) : "memory");
}

// Warp 0: issue layer l's phase-A copies (router rows by lane 0, the RMSNorm
// weight by lane 1, then the shared gate/up chunks).
__device__ void issue_A(const FusedParams& P, const FGeo& g, int l, const FSmem& S) {
  const FusedLayer& L = P.layers[l];
  const int d = P.d, E = P.E, f = P.f, lane = threadIdx.x & 31;
  fence_proxy_async();
  if (lane == 0) {
    // router rows [r0, r1) of rows 0..E (row E is the shared-gate vector)
    const int r0 = (int)blockIdx.x * g.rpc;
    int r1 = r0 + g.rpc;
    const int nrows = E + (L.sgate ? 1 : 0);
    if (r1 > nrows) r1 = nrows;
    const int nr = r1 > r0 ? r1 - r0 : 0;
    uint64_t* m = S.mR;
    mbar_expect_tx(S.mR, (uint32_t)nr * 2 * d);
    if (nr > 0) {
      const int nE = (r1 < E ? r1 : E) - r0;  // rows taken from the router matrix
      if (nE > 0) bulk_g2s(S.bufA, L.router + (size_t)r0 * d, (uint32_t)nE * 2 * d, m);
      if (nr > nE) bulk_g2s(S.bufA + (size_t)nE * 2 * d, L.sgate, 2 * d, m);
    }
  }
  if (lane == 1) {  // RMSNorm weight of the layer (stack mode)
    const bool has = P.stack && L.rho;
    mbar_expect_tx(S.mRho, has ? (uint32_t)d * 2 : 0u);
    if (has) bulk_g2s(S.rho, L.rho, d * 2, S.mRho);
  }
  // shared gate/up chunks, one piece per lane (see issue_B)
  static_assert(kMaxSC <= 8, "one instruction issues up to 8 chunks");
  {
    int b, e;
    s1_range(g, f, b, e);
    const int c = lane >> 2, piece = lane & 3;
    const Chunk ch = chunk_at(c < kMaxSC ? c : 0, b, e, f);
    uint64_t* m = &S.mS[c < kMaxSC ? c : 0];
    if (c < kMaxSC && piece == 0) mbar_expect_tx(m, (uint32_t)ch.n * g.unit);  // 0: completes empty
    __syncwarp();
    if (c < kMaxSC && ch.n > 0) {
      const int wq = g.wpr * 4, ws = g.gpr * 4;
      unsigned char* cb = S.bufA + s1_base(g, d) + (size_t)(ch.start - b) * g.unit;
      const int row = (piece & 1) ? f + ch.start : ch.start;  // gate rows, then up rows
      if (piece < 2)
        bulk_g2s(cb + piece * ch.n * wq, L.shared_q + (size_t)row * g.wpr, ch.n * wq, m);
      else
        bulk_g2s(cb + 2 * ch.n * wq + (piece - 2) * ch.n * ws,
              reinterpret_cast<const uint32_t*>(L.shared_sb) + (size_t)row * g.gpr, ch.n * ws, m);
    }
  }
  if (lane == 0) *S.apar = l & 1;
}

// One warp: issue layer l's phase-B copies (gate/up rows of the selected
// experts).
__device__ void issue_B(const FusedParams& P, const FGeo& g, int l, const FSmem& S, const int* s_idx) {
  const FusedLayer& L = P.layers[l];
  const int f = P.f, lane = threadIdx.x & 31;
  fence_proxy_async();
  // One copy per lane: lanes 4c..4c+3 issue chunk c's four pieces (gate rows,
  // up rows, their scale/bias rows), eight chunks per instruction. A copy
  // instruction costs its thread ~0.1 us to issue, so one lane per piece
  // issues fastest, and chunk-major order lets chunk 0 land first.
  int b, e;
  fsplit(P.K * f, blockIdx.x, g.nC, b, e);
  for (int c0 = 0; c0 < kMaxBC; c0 += 8) {
    const int c = c0 + (lane >> 2), piece = lane & 3;
    const Chunk ch = chunk_at(c, b, e, f);
    uint64_t* m = &S.mB[c];
    if (piece == 0) mbar_expect_tx(m, (uint32_t)ch.n * g.unit);  // 0: completes empty
    __syncwarp();
    if (ch.n > 0) {
      const int wq = g.wpr * 4, ws = g.gpr * 4;
      const int k = ch.start / f, r = ch.start - k * f;
      const int row = (piece & 1) ? f + r : r;  // gate rows, then up rows
      unsigned char* cb = S.bufB + (size_t)(ch.start - b) * g.unit;
      if (piece < 2)
        bulk_g2s(cb + piece * ch.n * wq, L.pool_q + (size_t)s_idx[k] * L.q_stride + (size_t)row * g.wpr, ch.n * wq,
                 m);
      else
        bulk_g2s(cb + 2 * ch.n * wq + (piece - 2) * ch.n * ws,
                 reinterpret_cast<const uint32_t*>(L.pool_sb + (size_t)s_idx[k] * L.sb_stride) + (size_t)row * g.gpr,
                 ch.n * ws, m);
    }
  }
  if (lane == 0) *S.bpar = l & 1;
}

// Phase C's shared-memory layout in bufB for rows [c_b, c_b + n) of d:
// q rows of slot k at k*n*wqf, scale/bias rows at (K+1)*n*wqf + k*n*wsf,
// partial results ys[k][r] after both.
struct CLayout {
  int n, wqf, wsf, f;
  __device__ size_t q(int k) const { return (size_t)k * n * wqf; }
  __device__ size_t sb(int K, int k) const { return (size_t)(K + 1) * n * wqf + (size_t)k * n * wsf; }
  __device__ size_t ys(int K) const { return ((size_t)(K + 1) * n * (wqf + wsf) + 15) & ~(size_t)15; }
  __device__ size_t hk(int K) const { return (ys(K) + (size_t)(K + 1) * n * 4 + 15) & ~(size_t)15; }
  __device__ size_t sth(int K) const { return (hk(K) + (size_t)(K + 1) * f * 4 + 15) & ~(size_t)15; }
};

// Warp 0: issue phase C's copies (the CTA's down rows of the K selected
// experts and of the shared expert) into bufB; lane k copies slot k.
template <int BITS>
__device__ void issue_C(const FusedParams& P, const FGeo& g, int l, const FSmem& S, const int* s_idx, int c_b,
                        const CLayout& cl) {
  const FusedLayer& L = P.layers[l];
  const int f = P.f, K = P.K, lane = threadIdx.x & 31;
  fence_proxy_async();
  if (lane == 0) mbar_expect_tx(S.mC, (uint32_t)((K + 1) * cl.n * (cl.wqf + cl.wsf)));
  __syncwarp();
  if (lane <= K && cl.n > 0) {
    const uint32_t* q;
    const uint16_t* sb;
    if (lane < K) {
      q = L.pool_q + (size_t)s_idx[lane] * L.q_stride;
      sb = L.pool_sb + (size_t)s_idx[lane] * L.sb_stride;
    } else {
      q = L.shared_q;
      sb = L.shared_sb;
    }
    q += 2 * (size_t)f * g.wpr + (size_t)c_b * (f * BITS / 32);
    sb += 2 * (size_t)f * g.gpr * 2 + (size_t)c_b * (f / kGroup) * 2;
    bulk_g2s(S.bufB + cl.q(lane), q, (uint32_t)cl.n * cl.wqf, S.mC);
    bulk_g2s(S.bufB + cl.sb(K, lane), sb, (uint32_t)cl.n * cl.wsf, S.mC);
  }
  if (lane == 0) *S.cpar = l & 1;
}

// Phase C's dot products: rows [0, cl.n) of the down matrices of slots
// 0..K (staged SwiGLU outputs of token k = slot k). The (slot, row group)
// work is cut into chunks of at most kCU row groups of one slot (as few
// chunks per slot as that allows, of near-equal size). A warp loads the
// slot's staged chunks for its part once, runs the chunk's rows as
// independent chains and reduces them together; ys[k * cl.n + r] = row r of
// slot k.
constexpr int kCU = 9;

template <int BITS>
__device__ __forceinline__ void down_rows(const unsigned char* buf, const CLayout& cl, int K, const XStage& sth,
                                          const RowGeo& rgf, float* ys, int warp, int lane) {
  using G = Geo<BITS>;
  const int nrows = cl.n;
  const int nrg = (nrows + rgf.RPP - 1) / rgf.RPP;
  const int cpk = (nrg + kCU - 1) / kCU;  // chunks per slot
  const int nch = cpk * (K + 1);
  const int lp = lane % rgf.LPR, rs = lane / rgf.LPR;
  const int rstep = rgf.RPP * cl.wqf, sstep = rgf.RPP * cl.wsf;
#pragma unroll 1
  for (int c = warp; c < nch; c += kFWarps) {
    const int k = c / cpk, ci = c - k * cpk;
    const int g0 = nrg * ci / cpk, g1 = nrg * (ci + 1) / cpk;  // at most kCU row groups
    uint4 xc[4 * G::kNch];
    uint2 xh[4 * G::kNch];
    load_part_x<BITS>(sth, k, 0, lp, rgf, xc, xh);
    const float2 pi = sth.partinfo[k * rgf.P + lp];
    const int r0 = g0 * rgf.RPP + rs;
    const unsigned char* qb = buf + cl.q(k) + (size_t)r0 * cl.wqf + lp * 16;
    const unsigned char* sbb = buf + cl.sb(K, k) + (size_t)r0 * cl.wsf + part_group<BITS>(lp) * 4;
    float v[kCU];
#pragma unroll
    for (int u = 0; u < kCU; ++u) {
      v[u] = 0.f;
      if (g0 + u < g1 && r0 + u * rgf.RPP < nrows) {
        const uint4 q = *reinterpret_cast<const uint4*>(qb + u * rstep);
        const uint32_t sbw = *reinterpret_cast<const uint32_t*>(sbb + u * sstep);
        v[u] = part_dot_x<BITS>(q, sbw, xc, xh, pi, 0.f);
      }
    }
    if (rgf.LPR >= 8) {
      float w8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w8[u] = v[u];
      const float y = row_reduce8(w8, rgf.LPR, lane);
      const int o1 = rgf.LPR >> 1, o2 = o1 >> 1, o3 = o2 >> 1;
      if ((lp & (o3 - 1)) == 0) {
        const int u = ((lp & o1) ? 4 : 0) + ((lp & o2) ? 2 : 0) + ((lp & o3) ? 1 : 0);
        const int rloc = r0 + u * rgf.RPP;
        if (g0 + u < g1 && rloc < nrows) ys[k * nrows + rloc] = y;
      }
#pragma unroll
      for (int u = 8; u < kCU; ++u) {
        const float y2 = row_reduce(v[u], rgf.LPR);
        const int rloc = r0 + u * rgf.RPP;
        if (lp == 0 && g0 + u < g1 && rloc < nrows) ys[k * nrows + rloc] = y2;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kCU; ++u) {
        const float y = row_reduce(v[u], rgf.LPR);
        const int rloc = r0 + u * rgf.RPP;
        if (lp == 0 && g0 + u < g1 && rloc < nrows) ys[k * nrows + rloc] = y;
      }
    }
  }
}

// --------------------------------------------------------------- the kernel
template <int BITS>
__global__ void __launch_bounds__(kFThreads, 1) k_fused_decode(const __grid_constant__ FusedParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int d = P.d, f = P.f, E = P.E, K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const FGeo g = fgeo(gridDim.x, d, f, E, K, BITS);
  Ctrl* ctrl = P.ctrl;
  const RowGeo rgd = row_geo(d, BITS);
  const RowGeo rgf = row_geo(f, BITS);

  // ---- shared memory
  const FLayout FL = flayout(g, d, f, K, BITS);
  FSmem S;
  S.mR = reinterpret_cast<uint64_t*>(smem);
  S.mRho = S.mR + 1;
  S.mC = S.mR + 2;
  S.mS = S.mR + 3;
  S.rho = reinterpret_cast<uint16_t*>(smem + FL.rho);
  S.mB = S.mS + kMaxSC;
  S.apar = reinterpret_cast<int*>(smem + FL.misc);
  S.bpar = S.apar + 1;
  S.cpar = S.apar + 52;
  int* s_idx = S.apar + 2;                              // [8]   ints 2..9
  float* s_w = reinterpret_cast<float*>(S.apar + 10);  // [9]   ints 10..18
  float* red = reinterpret_cast<float*>(S.apar + 20);  // [16]  ints 20..35
  float* s_l = reinterpret_cast<float*>(S.apar + 36);  // [9]   ints 36..44 (< 52)
  uint16_t* a_s = reinterpret_cast<uint16_t*>(smem + FL.a_s);
  const XStage sta = xstage_carve(smem + FL.sta, 1, d);
  S.bufA = smem + FL.bufA;
  S.bufB = smem + FL.bufB;
  // Stack mode: this CTA's rows [c_b, c_e) of the residual stream (the input
  // token before layer 0). The CTA writes the same rows every layer (and
  // thread t always row c_b + t), so the combine adds to this copy instead of
  // reading them back from L2 (20.96 -> 20.58 us per layer, 24-layer stack).
  float* hres = reinterpret_cast<float*>(smem + FL.hres);
  __shared__ float s_r;

  if (tid == 0) {
    mbar_init(S.mR, 1);
    mbar_init(S.mRho, 1);
    mbar_init(S.mC, 1);
    for (int j = 0; j < kMaxSC; ++j) mbar_init(&S.mS[j], 1);
    for (int j = 0; j < kMaxBC; ++j) mbar_init(&S.mB[j], 1);
    *S.apar = -1;
    *S.bpar = -1;
    *S.cpar = -1;
    fence_mbar_init();
  }
  if (P.stack) {  // the token's input rows of this CTA: the residual before layer 0
    int hb, he;
    fsplit(d, blockIdx.x, g.nC, hb, he);
    for (int k = hb + tid; k < he; k += kFThreads) hres[k - hb] = bf16f(P.x_in[k]);
  }
  __syncthreads();
  if (warp == 0) issue_A(P, g, 0, S);

  for (int l = 0; l < P.n_layers; ++l) {
    const FusedLayer& L = P.layers[l];
    const uint32_t par = (uint32_t)(l & 1);
    const bool has_gate = L.sgate != nullptr;
    stamp(P, l, 0);

    // ---------------- A0: layer input (RMSNorm of the residual in stack mode)
    if (P.stack) {
      if (l > 0 && !cta_wait(&ctrl->misc[4], g.nC * l, ctrl, P.timeout_ns, S)) return;
      stamp(P, l, 1);
      // one round trip: this thread's 8-element slices of the residual and of rho,
      // and (warp 0) the per-CTA sums of squares of the previous layer
      constexpr int kA0 = 2;  // slices per thread (d <= 8192)
      float hv[kA0][8];
      uint4 rv[kA0];
#pragma unroll
      for (int i = 0; i < kA0; ++i) {
        const int c = tid + i * kFThreads;
        rv[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[i][j] = 0.f;
        if (c < d / 8) {
          if (l == 0) {
            const uint4 xv = *reinterpret_cast<const uint4*>(P.x_in + 8 * c);
            hv[i][0] = bf16lo(xv.x); hv[i][1] = bf16hi(xv.x); hv[i][2] = bf16lo(xv.y); hv[i][3] = bf16hi(xv.y);
            hv[i][4] = bf16lo(xv.z); hv[i][5] = bf16hi(xv.z); hv[i][6] = bf16lo(xv.w); hv[i][7] = bf16hi(xv.w);
          } else {
            const float4 h0 = __ldcg(reinterpret_cast<const float4*>(P.h + 8 * c));
            const float4 h1 = __ldcg(reinterpret_cast<const float4*>(P.h + 8 * c + 4));
            hv[i][0] = h0.x; hv[i][1] = h0.y; hv[i][2] = h0.z; hv[i][3] = h0.w;
            hv[i][4] = h1.x; hv[i][5] = h1.y; hv[i][6] = h1.z; hv[i][7] = h1.w;
          }
        }
      }
      mbar_wait(S.mRho, par, ctrl, P.timeout_ns);
#pragma unroll
      for (int i = 0; i < kA0; ++i) {
        const int c = tid + i * kFThreads;
        if (c < d / 8) rv[i] = *reinterpret_cast<const uint4*>(S.rho + 8 * c);
      }
      if (l == 0) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kA0; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) ss = fmaf(hv[i][j], hv[i][j], ss);
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < kFWarps; ++w) s += red[w];
          s_r = 1.f / sqrtf(s / (float)d + P.eps);
        }
      } else if (warp == 0) {
        // the previous layer's per-CTA sums of squares: all loads in flight, then summed in order
        const float* part = P.part_ss + (l & 1) * g.nC;
        float s = 0.f;
        for (int c0 = 0; c0 < g.nC; c0 += 8 * 32) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = c0 + i * 32 + lane < g.nC ? __ldcg(part + c0 + i * 32 + lane) : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) s += v[i];
        }
        s = warp_sum(s);
        if (lane == 0) s_r = 1.f / sqrtf(s / (float)d + P.eps);
      }
      __syncthreads();
      const float r = s_r;
#pragma unroll
      for (int i = 0; i < kA0; ++i) {
        const int c = tid + i * kFThreads;
        if (c < d / 8) {
          const float rho[8] = {bf16lo(rv[i].x), bf16hi(rv[i].x), bf16lo(rv[i].y), bf16hi(rv[i].y),
                                bf16lo(rv[i].z), bf16hi(rv[i].z), bf16lo(rv[i].w), bf16hi(rv[i].w)};
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t lo = f2bf((hv[i][2 * j] * r) * rho[2 * j]);
            const uint32_t hi = f2bf((hv[i][2 * j + 1] * r) * rho[2 * j + 1]);
            o[j] = lo | (hi << 16);
          }
          *reinterpret_cast<uint4*>(a_s + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    } else {
      for (int k = tid; k < d / 8; k += kFThreads)
        reinterpret_cast<uint4*>(a_s)[k] = reinterpret_cast<const uint4*>(P.x_in)[k];
    }
    __syncthreads();
    stamp(P, l, 2);

    // ---------------- A1: router rows (in bufA)
    {
      const int rloc = warp / g.qr, qtr = warp - rloc * g.qr;
      const int row = (int)blockIdx.x * g.rpc + rloc;
      const bool valid = rloc < g.rpc && row < E + (has_gate ? 1 : 0);
      float v = 0.f;
      if (valid) {
        mbar_wait(S.mR, par, ctrl, P.timeout_ns);
        const int c0 = qtr * (d / g.qr);
        v = router_dot(reinterpret_cast<const uint16_t*>(S.bufA) + (size_t)rloc * d, a_s, c0, d / g.qr / 256, lane);
      }
      if (lane == 0) red[warp] = v;
      __syncthreads();
      if (valid && qtr == 0 && lane == 0) {
        float s = 0.f;
        for (int q = 0; q < g.qr; ++q) s += red[warp + q];
        // one 64-bit word {value, tag}: a reader that sees the tag sees the
        // value, so the exchange needs no fence and no counter
        st_relaxed_u64(P.ltag + row, ((unsigned long long)(l + 1) << 32) | __float_as_uint(s));
      }
    }
    stamp(P, l, 3);
    {  // Staged integer copy of the input for the gate/up rows, while the
       // logits of the other CTAs arrive: fp32 copy in bufB (free until the
       // selection), then staged.
      float* af = reinterpret_cast<float*>(S.bufB);
      for (int k = tid; k < d; k += kFThreads) af[k] = bf16f(a_s[k]);
      __syncthreads();
      stage_f32<BITS>(af, d, 1, d, sta);
    }
    stamp(P, l, 12);

    // ---------------- selection: every CTA selects from the complete logits
    {
      // Each thread polls its logits' words until they carry this layer's tag
      // (bounded: an abort elsewhere or the time limit ends the wait; the
      // exchange is described at the top of the file).
      float* lg_s = reinterpret_cast<float*>(S.bufB);  // bufB is free until the B copies
      const unsigned tag = (unsigned)l + 1u;  // the words are zero when a launch starts
      const int nrows = E + (has_gate ? 1 : 0);
      __shared__ int s_fail;
      if (tid == 0) s_fail = 0;
      __syncthreads();
      for (int e = tid; e < nrows; e += kFThreads) {
        unsigned long long v = ld_relaxed_u64(P.ltag + e);
        if ((unsigned)(v >> 32) != tag) {
          const unsigned long long t0 = globaltimer();
          long long it = 0;
          while ((unsigned)((v = ld_relaxed_u64(P.ltag + e)) >> 32) != tag) {
            if ((++it & 31) == 0) {
              if (aborted(ctrl)) {
                s_fail = 1;
                break;
              }
              if (it > kMaxSpin || (long long)(globaltimer() - t0) > P.timeout_ns) {
                raise_timeout(ctrl);
                s_fail = 1;
                break;
              }
            }
          }
        }
        lg_s[e] = __uint_as_float((unsigned)v);
      }
      __syncthreads();
      if (s_fail) {
        if (tid == 0) drain_copies(S);
        return;
      }
      stamp(P, l, 5);
      block_topk_select(lg_s, reinterpret_cast<int*>(lg_s + ((E + 4) & ~3)), E, K, has_gate, s_idx, s_l);
      stamp(P, l, 11);
    }

    // ---------------- B: the selected experts' gate/up units (in bufB)
    if (warp == kFWarps - 1) issue_B(P, g, l, S, s_idx);  // the last warp: its phase-B units (if any) come last
    if (warp == 0) {  // the routing weights (used by the combine) while phase B's copies start
      block_topk_weights(s_l, K, has_gate, s_w);
      __syncwarp();
      if (blockIdx.x == 0 && lane < K) {
        if (P.idx_out) P.idx_out[l * K + lane] = s_idx[lane];
        if (P.w_out) P.w_out[l * K + lane] = s_w[lane];
      }
      if (blockIdx.x == 0 && lane == 0 && P.gamma_out) P.gamma_out[l] = s_w[K];
    }
    {
      // The shared expert's gate/up units (phase A's data, in bufA) do not
      // gate the selection, so they run here, while phase B's rows stream in;
      // they go to the last warps, whose phase-B chunks land last.
      int b, e;
      s1_range(g, f, b, e);
      run_units<BITS>(S.bufA + s1_base(g, d), b, e, f, S.mS, par, ctrl, P.timeout_ns, sta, g,
                      P.hk + (size_t)K * f + b, kFWarps - 1 - warp, lane);
      stamp(P, l, 4);
      fsplit(K * f, blockIdx.x, g.nC, b, e);
      run_units<BITS>(S.bufB, b, e, f, S.mB, par, ctrl, P.timeout_ns, sta, g, P.hk + b, warp, lane);  // unit k*f + row
    }
    stamp(P, l, 6);
    // Phase C: this CTA's output rows [c_b, c_e). Once every warp is done with
    // bufB, warp 0 streams the down rows of the K+1 experts into it; they land
    // during the grid-wide wait. The next layer's phase-A data (into bufA)
    // follows once the wait is over, so that it does not slow the exchange.
    int c_b, c_e;
    fsplit(d, blockIdx.x, g.nC, c_b, c_e);
    CLayout cl;
    cl.n = c_e - c_b;
    cl.wqf = f * BITS / 8;
    cl.wsf = (f / kGroup) * 4;
    cl.f = f;
    const XStage sth = xstage_carve(S.bufB + cl.sth(K), K + 1, f);  // after the gathered fp32 copy
    cta_arrive(&ctrl->misc[3]);
    if (warp == 0) issue_C<BITS>(P, g, l, S, s_idx, c_b, cl);

    // ---------------- C: down rows + combine (+ residual)
    if (!cta_wait(&ctrl->misc[3], g.nC * (l + 1), ctrl, P.timeout_ns, S)) return;
    stamp(P, l, 7);
    if (warp == 0 && l + 1 < P.n_layers) issue_A(P, g, l + 1, S);  // lands during phase C and the next exchange
    {
      {  // the SwiGLU outputs of every CTA, through L2: all loads in flight, then staged
        float4* hks = reinterpret_cast<float4*>(S.bufB + cl.hk(K));
        const float4* src = reinterpret_cast<const float4*>(P.hk);
        const int n4 = (K + 1) * f / 4;
        for (int i0 = tid; i0 < n4; i0 += 4 * kFThreads) {
          float4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (i0 + j * kFThreads < n4) v[j] = __ldcg(src + i0 + j * kFThreads);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (i0 + j * kFThreads < n4) hks[i0 + j * kFThreads] = v[j];
        }
        __syncthreads();
        stage_x24_pairs<BITS>(StridedSrc<float>{reinterpret_cast<const float*>(hks), f}, K + 1, f, sth);
      }
      stamp(P, l, 13);
      mbar_wait(S.mC, par, ctrl, P.timeout_ns);
      stamp(P, l, 9);
      float* ys = reinterpret_cast<float*>(S.bufB + cl.ys(K));
      down_rows<BITS>(S.bufB, cl, K, sth, rgf, ys, warp, lane);
      const int nrows = cl.n;
      __syncthreads();
      stamp(P, l, 10);
      // combine in fixed order: routed experts k = 0..K-1, then the shared expert (k = K)
      float ss = 0.f;
      for (int rl = tid; rl < nrows; rl += kFThreads) {
        const int row = c_b + rl;
        float o = 0.f;
        for (int k = 0; k <= K; ++k) o = fmaf(s_w[k], ys[k * nrows + rl], o);
        if (P.stack) {
          const float hv = hres[rl] + o;
          P.h[row] = hv;
          hres[rl] = hv;
          ss = fmaf(hv, hv, ss);
        } else {
          if (P.out) P.out[row] = f2bf(o);
          if (P.out_f32) P.out_f32[row] = o;
        }
      }
      stamp(P, l, 14);
      if (P.stack) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < kFWarps; ++w) s += red[w];
          P.part_ss[((l + 1) & 1) * g.nC + blockIdx.x] = s;
        }
      }
    }
    stamp(P, l, 8);
    cta_arrive(&ctrl->misc[4]);
  }

  // ---------------- stack output: x_next = bf16(rmsnorm(h)), h_out
  if (P.stack) {
    if (!cta_wait(&ctrl->misc[4], g.nC * P.n_layers, ctrl, P.timeout_ns, S)) return;
    if (warp == 0) {
      const float* part = P.part_ss + (P.n_layers & 1) * g.nC;
      float s = 0.f;
      for (int c = lane; c < g.nC; c += 32) s += __ldcg(part + c);
      s = warp_sum(s);
      if (lane == 0) s_r = 1.f / sqrtf(s / (float)d + P.eps);
    }
    __syncthreads();
    int b, e;
    fsplit(d, blockIdx.x, g.nC, b, e);
    for (int k = b + tid; k < e; k += kFThreads) {
      const float hv = hres[k - b];  // written by this thread in the last layer's combine
      if (P.x_next) P.x_next[k] = f2bf(hv * s_r);
      if (P.h_out) P.h_out[k] = hv;
    }
  }
  // the last CTA out resets the counters and clears the tagged logits for the
  // next launch (every other CTA has read them by now)
  __syncthreads();
  __shared__ int s_last;
  int prev = 0;
  if (tid == 0) {
    prev = atomicAdd(&ctrl->misc[5], 1);
    s_last = prev == g.nC - 1;
  }
  __syncthreads();
  if (s_last)
    for (int e = tid; e <= E; e += kFThreads) P.ltag[e] = 0ull;
  if (tid == 0 && prev == g.nC - 1) {
    for (int i = 1; i <= 5; ++i) ctrl->misc[i] = 0;
    __threadfence();
  }
}

// --------------------------------------------------------------- wait self-test
// Two CTAs wait on a counter nothing increments, with a short limit: the
// bounded wait must give up, write BGQ_ERR_TIMEOUT and return. Exercises the
// same grid-wide wait the decode kernel uses, without faulting anything.
__global__ void k_wait_selftest(Ctrl* ctrl, long long timeout_ns) {
  FSmem S{};
  __shared__ int par[3];
  if (threadIdx.x == 0) {
    par[0] = -1;
    par[1] = -1;
    par[2] = -1;
  }
  __syncthreads();
  S.apar = &par[0];
  S.bpar = &par[1];
  S.cpar = &par[2];
  if (!cta_wait(&ctrl->misc[6], 1 << 30, ctrl, timeout_ns, S)) return;
  if (threadIdx.x == 0) atomicExch(&ctrl->status, BGQ_OK);  // not reached: nothing sets misc[6]
}

cudaError_t launch_wait_selftest(Ctrl* ctrl, long long timeout_ns, cudaStream_t s) {
  k_wait_selftest<<<2, 64, 0, s>>>(ctrl, timeout_ns);
  return cudaGetLastError();
}

// --------------------------------------------------------------- host side
static size_t fused_smem_for(const FGeo& g, int d, int f, int K, int bits) {
  return flayout(g, d, f, K, bits).total;
}

size_t fused_smem_bytes(int d, int f, int K, int bits) {
  FGeo g = fgeo(num_sms(), d, f, 1024, K, bits);
  return fused_smem_for(g, d, f, K, bits);
}

bool fused_supported(int d, int f, int E, int K, int bits) {
  if (K < 1 || K > 8 || E < K || E > 1024) return false;
  if (d % 256 || f % 256) return false;  // scale/bias rows of 16-byte multiples (bulk copies)
  if (d > 2048 && d % 1024) return false;  // router slices of 1024 columns, or one slice of <= 2048
  const int Pd = d * bits / 128, Pf = f * bits / 128;
  if (Pd < 32 || Pd % 32 || Pd / 32 > 4) return false;  // d-rows: all lanes, <= 4 parts each
  if (Pf < 1 || Pf > 32 || 32 % Pf) return false;       // f-rows: one part per lane
  const int nC = num_sms();
  FGeo g = fgeo(nC, d, f, E, K, bits);
  if (g.nRouter > nC) return false;  // every router row owned by one CTA
  if (g.nBmax > kMaxB) return false;
  // bulk-copy chunks per CTA
  for (int c = 0; c < nC; ++c) {
    int b, e;
    fsplit(K * f, c, nC, b, e);
    int start = b, nch = 0;
    while (start < e) {
      int lim = start + kCH < e ? start + kCH : e;
      int seg = (start / f + 1) * f;
      if (seg < lim) lim = seg;
      start = lim;
      ++nch;
    }
    if (nch > kMaxBC) return false;
  }
  // largest shared gate/up range of any CTA
  int mx = g.s1_nr;
  const int n_nr = nC - g.nRouter;
  const int rest0 = g.s1_nr > 0 ? n_nr * g.s1_nr : 0;
  const int nparts = g.s1_nr > 0 ? g.nRouter : nC;
  for (int c = 0; c < nparts; ++c) {
    int b, e;
    fsplit(f - rest0, c, nparts, b, e);
    if (e - b > mx) mx = e - b;
  }
  if (mx > kMaxS1 || (mx + kCH - 1) / kCH > kMaxSC) return false;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  return fused_smem_for(g, d, f, K, bits) + 1024 <= (size_t)optin;
}

cudaError_t launch_fused(const FusedParams& P, int bits, cudaStream_t s) {
  const int nC = num_sms();
  FGeo g = fgeo(nC, P.d, P.f, P.E, P.K, bits);
  size_t sm = fused_smem_for(g, P.d, P.f, P.K, bits);
  void* kern = bits == 4 ? (void*)k_fused_decode<4> : (void*)k_fused_decode<2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&P};
  return cudaLaunchCooperativeKernel(kern, dim3(nC), dim3(kFThreads), args, sm, s);
}

}  // namespace bgq
