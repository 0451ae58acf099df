// fused.cu — one persistent kernel for batch-1 decode: a whole token through
// one MoE layer or a stack of layers per launch.
//
// Flash-MoE page, section "架构设计：SSD当显存用": per token and layer the path
// is routing logits -> softmax + top-K -> the selected experts' forward pass
// -> combine (-> norm). At batch 1 every step is a matrix-vector product whose
// weights are read exactly once, so a layer is bound by HBM bandwidth and by
// the latency of its dependent steps. One cooperative launch with one CTA per
// SM keeps the token on chip and replaces kernel boundaries by grid-wide
// exchanges. Per layer, every CTA:
//
//   A  normalises the residual (stack mode: RMSNorm with the layer's weight,
//      rounded to bf16 as the layer input), computes its router rows (copied
//      into region B during the previous layer) and publishes those logits as
//      tagged words, then stages the input as 24-bit fixed point;
//   S  once every logit carries the layer's tag, selects the same top-K as
//      every other CTA and at once requests its share of the selected
//      experts' gate/up rows (region B);
//   B  computes its share of the shared expert's gate/up rows (region A,
//      copied during the previous layer) while those land, then requests its
//      output rows of all K + 1 down matrices into region A (free again), then
//      computes its selected gate/up rows as they land and publishes the
//      SwiGLU outputs; counts itself in the SwiGLU counter;
//   C  after that counter, requests the next layer's router rows (region B),
//      stages every SwiGLU output straight from L2, computes its output rows
//      of the K + 1 down matrices (landed behind the gate/up rows), requests
//      the next layer's shared gate/up rows (region A), combines the rows in a
//      fixed order and adds the residual, then counts itself in the residual
//      counter.
//
// The down rows depend only on the selection, so they follow the gate/up rows
// into memory at once and have landed before the SwiGLU exchange starts;
// requested only after phase B, they and the exchange's counter polls
// competed for memory on the critical path.
//
// Code size matters as much as the data path here: every phase's code runs
// once per layer, so a kernel larger than the instruction cache pays a miss
// at every phase. The work split and the shared-memory layout are computed on
// the host (FGeo), the chunk tables once per launch, waits are compact loops,
// and the paths that only run on a timeout are out of line.
//
// Exchanges. The logits (2 KB) go as 64-bit {value, layer + 1} words written
// with relaxed stores and polled by every thread for its share: a reader that
// sees the tag sees the value, so no fence and no counter are needed (the
// words are zero at every launch's start, the last CTA out clears them). The
// SwiGLU outputs and the residual use counters: a CTA's release reduction
// after a block barrier, thread 0 polling with acquire loads.
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
constexpr int kCH = 7;       // units per bulk-copy chunk (one mbarrier per chunk)
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
__device__ __noinline__ void raise_timeout(Ctrl* ctrl) {
  atomicExch(&ctrl->status, BGQ_ERR_TIMEOUT);
  atomicExch(&ctrl->misc[0], 1);
}

// Bounded wait for mbarrier phase `parity`; false on timeout or abort. The
// loop is out of line; callers test the phase first (mbar_wait).
__device__ __noinline__ bool mbar_wait_loop(uint64_t* m, uint32_t parity, Ctrl* ctrl, long long timeout_ns) {
  unsigned long long t0 = 0;
  for (int it = 1; !mbar_try_wait(m, parity); ++it) {
    if ((it & 31) == 0) {
      const unsigned long long t = globaltimer();
      if (t0 == 0) t0 = t;
      if (aborted(ctrl)) return false;
      if ((long long)(t - t0) > timeout_ns || it > (int)kMaxSpin) {
        raise_timeout(ctrl);
        return false;
      }
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity, Ctrl* ctrl, long long timeout_ns) {
  return mbar_try_wait(m, parity) || mbar_wait_loop(m, parity, ctrl, timeout_ns);
}

// --------------------------------------------------------------- geometry
__host__ __device__ inline void fsplit(int n, int part, int nparts, int& b, int& e) {
  b = n * part / nparts;  // n * nparts < 2^31 for every split here
  e = n * (part + 1) / nparts;
}
__host__ __device__ inline int up128(int n) { return (n + 127) & ~127; }
__host__ __device__ inline int up16(int n) { return (n + 15) & ~15; }

// Shared-memory layout: [mbarriers][misc ints][a_s: layer input, bf16]
// [sta: staged layer input][hres: this CTA's residual rows][A][B].
// A: the shared expert's gate/up units; once they are computed, the down rows
//    of the K + 1 experts and their partial results.
// B: the router rows; the selection's logits and scratch; the selected
//    gate/up units; after phase B, the next layer's router rows and the
//    staged SwiGLU outputs.
constexpr int kMiscInts = 256;
static FGeo fused_geo(int nC, int d, int f, int E, int K, int bits) {
  FGeo g{};
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
    const double total = (double)(E + 1) * 2 * d + (double)f * g.unit;
    int a = (int)(total / nC / g.unit + 0.5);
    if (a * n_nr > f) a = f / n_nr;
    if (a > kMaxS1) a = kMaxS1;
    g.s1_nr = a < 0 ? 0 : a;
  }
  g.s1_rest0 = g.s1_nr > 0 ? n_nr * g.s1_nr : 0;
  g.s1_nparts = g.s1_nr > 0 ? g.nRouter : nC;
  const int s1_router = (f - g.s1_rest0 + g.s1_nparts - 1) / g.s1_nparts;
  const int s1_max = s1_router > g.s1_nr ? s1_router : g.s1_nr;
  g.rows_c = (d + nC - 1) / nC;
  g.wqf = f * bits / 8;
  g.wsf = (f / kGroup) * 4;
  const int a_c = up16((K + 1) * g.rows_c * (g.wqf + g.wsf)) + (K + 1) * g.rows_c * 4;
  g.a_bytes = s1_max * g.unit > a_c ? s1_max * g.unit : a_c;
  const int b_units = g.nBmax * g.unit;
  const int b_c = up16(g.rpc * 2 * d) + (int)xstage_bytes(K + 1, f, bits);
  const int b_sel = (((E + 4) & ~3) + topk_scratch_ints(E)) * 4;
  g.b_bytes = b_units > b_c ? b_units : b_c;
  if (g.b_bytes < b_sel) g.b_bytes = b_sel;
  int o = 256;  // mbarriers
  g.o_misc = o;
  o += up128(kMiscInts * 4);
  g.o_as = o;
  o += up128(d * 2);
  g.o_sta = o;
  o += up128((int)xstage_bytes(1, d, bits));
  g.o_hres = o;
  o += up128(g.rows_c * 4);
  g.o_a = o;
  o += up128(g.a_bytes);
  g.o_b = o;
  o += up128(g.b_bytes);
  g.total = o;
  return g;
}

// Misc ints (shared memory): parities of the last issued copies, this CTA's
// ranges and chunk tables, the selection and small reductions.
enum MiscSlot {
  kApar = 0, kBpar, kCpar, kS1b, kS1e, kNS, kBb, kBe, kNB, kCb, kCe, kFail, kLast, kSpar,
  kIdx = 16,        // [8]
  kW = 24,          // [9] floats: routing weights, then gamma
  kL = 40,          // [9] floats: selected logits, then the shared-gate logit
  kRed = 56,        // [16] floats
  kR = 72,          // float: 1 / rms
  kChS = 80,        // [kMaxSC][2]: shared chunks (start, n)
  kChB = 96,        // [kMaxBC][2]: selected chunks (start, n)
};

// Chunks of units [b, e): at most kCH units, never across a multiple of seg
// (an expert boundary). Returns the number of chunks.
__device__ int make_chunks(int b, int e, int seg, int maxc, int* tab) {
  int n = 0;
  for (int start = b; start < e && n < maxc; ++n) {
    int lim = min(start + kCH, e);
    lim = min(lim, (start / seg + 1) * seg);
    tab[2 * n] = start;
    tab[2 * n + 1] = lim - start;
    start = lim;
  }
  return n;
}
__device__ __forceinline__ int chunk_find(const int* tab, int nch, int u) {
  int c = 0;
  while (c + 1 < nch && u >= tab[2 * (c + 1)]) ++c;
  return c;
}

// --------------------------------------------------------------- compute helpers
// NR integer dot products of one 128-bit part each (codes q[i], scale/bias
// sbw[i]) against the same staged input part (slot `slot`, lanes of a row
// LPR apart; part info pi): acc[i] += s_i*2^-sh*sum(q_i*X) + b_i*2^-sh*sum(X).
// The input bytes are loaded one code word at a time and shared by all rows.
template <int BITS, int NR>
__device__ __forceinline__ void part_dots(const uint4 (&q)[NR], const uint32_t (&sbw)[NR], const XStage& st, int slot,
                                          int LPR, const float2 pi, float (&acc)[NR]) {
  using G = Geo<BITS>;
  uint32_t L0[NR], M0[NR], L1[NR], M1[NR];
  int H0[NR], H1[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    L0[i] = M0[i] = L1[i] = M1[i] = 0u;
    H0[i] = H1[i] = 0;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int ch = 0; ch < G::kNch; ++ch) {
      const int s = slot + (c * G::kNch + ch) * LPR;
      const uint4 x = st.chunks[s];
      const uint2 xh = st.hib[s];
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        const uint32_t w = c == 0 ? q[i].x : c == 1 ? q[i].y : c == 2 ? q[i].z : q[i].w;
        uint32_t v0, v1;
        if (BITS == 4) {  // odd codes stay in the high nibbles (16x), divided out at the end
          v0 = w & 0x0f0f0f0fu;
          v1 = w & 0xf0f0f0f0u;
        } else {
          v0 = (w >> (BITS * (2 * ch))) & G::kByteMask;
          v1 = (w >> (BITS * (2 * ch + 1))) & G::kByteMask;
        }
        L0[i] = dp4a_uu(v0, x.x, L0[i]);
        M0[i] = dp4a_uu(v0, x.y, M0[i]);
        H0[i] = dp4a_us(v0, xh.x, H0[i]);
        L1[i] = dp4a_uu(v1, x.z, L1[i]);
        M1[i] = dp4a_uu(v1, x.w, M1[i]);
        H1[i] = dp4a_us(v1, xh.y, H1[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    int lo, hi;
    if (BITS == 4) {
      lo = (int)(L0[i] + (L1[i] >> 4)) + (int)(M0[i] + (M1[i] >> 4)) * 256;
      hi = H0[i] + (H1[i] >> 4);
    } else {
      lo = (int)(L0[i] + L1[i]) + (int)(M0[i] + M1[i]) * 256;
      hi = H0[i] + H1[i];
    }
    const float A = fmaf((float)hi, 65536.f, (float)lo);
    acc[i] = fmaf(bf16lo(sbw[i]) * pi.x, A, fmaf(bf16hi(sbw[i]), pi.y, acc[i]));
  }
}

// Gate and up rows of two units (in shared memory) against the staged layer
// input: four dot products that share every input load. Unit i is at position
// p_i of a chunk of n_i units starting at c_i. Lane l reads part it*32 + l.
// Returns silu(gate) * up of unit 0 in lane 0 and of unit 1 in lane 16.
template <int BITS>
__device__ __noinline__ float units_gateup2(const unsigned char* c0, int n0, int p0, const unsigned char* c1, int n1,
                                            int p1, const XStage st, const FGeo g, int lane) {
  const int wq = g.wpr * 4, ws = g.gpr * 4;
  const uint4* qg0 = reinterpret_cast<const uint4*>(c0 + p0 * wq);
  const uint4* qu0 = reinterpret_cast<const uint4*>(c0 + (n0 + p0) * wq);
  const uint32_t* sg0 = reinterpret_cast<const uint32_t*>(c0 + 2 * n0 * wq + p0 * ws);
  const uint32_t* su0 = reinterpret_cast<const uint32_t*>(c0 + 2 * n0 * wq + (n0 + p0) * ws);
  const uint4* qg1 = reinterpret_cast<const uint4*>(c1 + p1 * wq);
  const uint4* qu1 = reinterpret_cast<const uint4*>(c1 + (n1 + p1) * wq);
  const uint32_t* sg1 = reinterpret_cast<const uint32_t*>(c1 + 2 * n1 * wq + p1 * ws);
  const uint32_t* su1 = reinterpret_cast<const uint32_t*>(c1 + 2 * n1 * wq + (n1 + p1) * ws);
  float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int it = 0; it < g.nit_d; ++it) {
    const int p = it * 32 + lane, pg = part_group<BITS>(p);
    const uint4 q[4] = {qg0[p], qu0[p], qg1[p], qu1[p]};
    const uint32_t sbw[4] = {sg0[pg], su0[pg], sg1[pg], su1[pg]};
    part_dots<BITS, 4>(q, sbw, st, it * 4 * Geo<BITS>::kNch * 32 + lane, 32, st.partinfo[p], v);
  }
  // lanes 0-7: gate 0, 8-15: up 0, 16-23: gate 1, 24-31: up 1 (bit-identical to warp_sum)
  const float r = row_reduce4(v, 32, lane);
  const float up = __shfl_down_sync(kFull, r, 8);
  return r / (1.f + expf(-r)) * up;
}

// Units [b, e) of a phase, in chunks tab[0..nch) (chunk c complete on
// mbars[c]), two per warp: hk_dst[j] = silu(gate) * up of unit b + j. An odd
// last unit is computed twice, written once. `wslot` is the warp's slot.
template <int BITS>
__device__ __forceinline__ void run_units(const unsigned char* base, int b, int e, const int* tab, int nch,
                                          uint64_t* mbars, uint32_t par, Ctrl* ctrl, long long timeout_ns,
                                          const XStage& st, const FGeo& g, float* hk_dst, int wslot, int lane) {
  const int nu = e - b;
  for (int j0 = 2 * wslot; j0 < nu; j0 += 2 * kFWarps) {
    const int j1 = min(j0 + 1, nu - 1);
    const int c0 = chunk_find(tab, nch, b + j0), c1 = chunk_find(tab, nch, b + j1);
    mbar_wait(&mbars[c0], par, ctrl, timeout_ns);
    if (c1 != c0) mbar_wait(&mbars[c1], par, ctrl, timeout_ns);
    const int s0 = tab[2 * c0], s1 = tab[2 * c1];
    const float h = units_gateup2<BITS>(base + (size_t)(s0 - b) * g.unit, tab[2 * c0 + 1], b + j0 - s0,
                                        base + (size_t)(s1 - b) * g.unit, tab[2 * c1 + 1], b + j1 - s1, st, g, lane);
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

// Event ev of layer l, stamped by thread 0 (events 14, 15: by the thread
// that calls; only in the traced instantiation, so that the production kernel
// carries none of this code).
template <bool TRACE>
__device__ __forceinline__ void stamp(const FusedParams& P, int l, int ev) {
  if (TRACE && (threadIdx.x == 0 || ev >= 14))
    P.trace[((size_t)l * gridDim.x + blockIdx.x) * kTraceEvents + ev] = globaltimer();
}

// Shared-memory state of the kernel.
struct FSmem {
  uint64_t* mR;  // router rows
  uint64_t* mC;  // down rows of phase C
  uint64_t* mS;  // [kMaxSC] shared gate/up chunks
  uint64_t* mB;  // [kMaxBC] selected gate/up chunks
  int* misc;
  unsigned char* A;
  unsigned char* B;
};

// Thread 0: wait (bounded) for every bulk copy this CTA still has in flight.
__device__ __noinline__ void drain_copies(const FSmem& S) {
  const unsigned long long t0 = globaltimer();
  const int ap = S.misc[kApar], sp = S.misc[kSpar], bp = S.misc[kBpar], cp = S.misc[kCpar];
  auto drain = [&](uint64_t* m, int par) {
    while (!mbar_try_wait(m, (uint32_t)par) && (long long)(globaltimer() - t0) < kDrainNs) {
    }
  };
  if (cp >= 0) drain(S.mC, cp);
  if (ap >= 0) drain(S.mR, ap);
  if (sp >= 0)
    for (int j = 0; j < S.misc[kNS]; ++j) drain(&S.mS[j], sp);
  if (bp >= 0)
    for (int j = 0; j < S.misc[kNB]; ++j) drain(&S.mB[j], bp);
}

// Grid-wide wait: thread 0 waits until *p >= target. False for the whole CTA
// on abort or timeout (after thread 0 drained the CTA's copies in flight).
__device__ __noinline__ bool cta_wait(const int* p, int target, Ctrl* ctrl, long long timeout_ns,
                                      const FSmem& S) {
  if (threadIdx.x == 0) {
    int ok = 1;
    unsigned long long t0 = 0;
    for (int it = 1; ld_acquire(p) < target; ++it) {
      if (it > 16) __nanosleep(32);
      if ((it & 15) == 0) {
        const unsigned long long t = globaltimer();
        if (t0 == 0) t0 = t;
        if (aborted(ctrl)) {
          ok = 0;
          break;
        }
        if ((long long)(t - t0) > timeout_ns || it > (int)kMaxSpin) {
          raise_timeout(ctrl);
          ok = 0;
          break;
        }
      }
    }
    if (ok && aborted(ctrl)) ok = 0;
    if (!ok) drain_copies(S);
    S.misc[kFail] = !ok;
  }
  __syncthreads();
  return S.misc[kFail] == 0;
}

// All threads: publish this CTA's global writes, then count it in *p
// (block barrier, then one release reduction by thread 0).
__device__ __forceinline__ void cta_arrive(int* p) {
  __syncthreads();
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p) : "memory");
}

// Lane 0 of warp 0: issue layer l's router rows into B (row E is the
// shared-gate vector).
__device__ void issue_router(const FusedParams& P, int l, const FSmem& S) {
  const FGeo& g = P.g;
  const FusedLayer& L = P.layers[l];
  const int d = P.d, E = P.E;
  fence_proxy_async();
  const int r0 = (int)blockIdx.x * g.rpc;
  const int nrows = E + (L.sgate ? 1 : 0);
  const int r1 = min(r0 + g.rpc, nrows);
  const int nr = r1 > r0 ? r1 - r0 : 0;
  mbar_expect_tx(S.mR, (uint32_t)nr * 2 * d);  // 0 bytes: the phase completes at once
  if (nr > 0) {
    const int nE = min(r1, E) - r0;  // rows taken from the router matrix
    if (nE > 0) bulk_g2s(S.B, L.router + (size_t)r0 * d, (uint32_t)nE * 2 * d, S.mR);
    if (nr > nE) bulk_g2s(S.B + (size_t)nE * 2 * d, L.sgate, 2 * d, S.mR);
  }
  S.misc[kApar] = l & 1;
}

// Warp 0: issue layer l's shared gate/up chunks into A, one piece (gate
// rows, up rows, their scale/bias rows) per lane.
__device__ void issue_shared(const FusedParams& P, int l, const FSmem& S) {
  const FGeo& g = P.g;
  const FusedLayer& L = P.layers[l];
  const int f = P.f, lane = threadIdx.x & 31;
  const int c = lane >> 2, piece = lane & 3;
  const int nS = S.misc[kNS], b = S.misc[kS1b];
  fence_proxy_async();
  if (c < nS) {
    const int start = S.misc[kChS + 2 * c], n = S.misc[kChS + 2 * c + 1];
    uint64_t* m = &S.mS[c];
    if (piece == 0) mbar_expect_tx(m, (uint32_t)n * g.unit);
    __syncwarp(0xfu << (4 * c));
    const int wq = g.wpr * 4, ws = g.gpr * 4;
    unsigned char* cb = S.A + (size_t)(start - b) * g.unit;
    const int row = (piece & 1) ? f + start : start;  // gate rows, then up rows
    if (piece < 2)
      bulk_g2s(cb + piece * n * wq, L.shared_q + (size_t)row * g.wpr, n * wq, m);
    else
      bulk_g2s(cb + 2 * n * wq + (piece - 2) * n * ws,
               reinterpret_cast<const uint32_t*>(L.shared_sb) + (size_t)row * g.gpr, n * ws, m);
  }
  if (lane == 0) S.misc[kSpar] = l & 1;
}

// Warp 15: issue layer l's phase-B copies into B (gate/up rows of the selected
// experts), chunk-major so that chunk 0 lands first; one piece per lane.
__device__ void issue_B(const FusedParams& P, int l, const FSmem& S, int cb0, int cb1) {
  const FGeo& g = P.g;
  const FusedLayer& L = P.layers[l];
  const int f = P.f, lane = threadIdx.x & 31;
  const int b = S.misc[kBb];
  const int* s_idx = S.misc + kIdx;
  fence_proxy_async();
#pragma unroll 1
  for (int c0 = cb0; c0 < cb1; c0 += 8) {
    const int c = c0 + (lane >> 2), piece = lane & 3;
    if (c < cb1) {
      const int start = S.misc[kChB + 2 * c], n = S.misc[kChB + 2 * c + 1];
      uint64_t* m = &S.mB[c];
      if (piece == 0) mbar_expect_tx(m, (uint32_t)n * g.unit);
      __syncwarp(0xfu << (lane & 28));
      const int wq = g.wpr * 4, ws = g.gpr * 4;
      const int k = start / f, r = start - k * f;  // expert slot, row
      const int row = (piece & 1) ? f + r : r;
      unsigned char* cb = S.B + (size_t)(start - b) * g.unit;
      if (piece < 2)
        bulk_g2s(cb + piece * n * wq, L.pool_q + (size_t)s_idx[k] * L.q_stride + (size_t)row * g.wpr, n * wq, m);
      else
        bulk_g2s(cb + 2 * n * wq + (piece - 2) * n * ws,
                 reinterpret_cast<const uint32_t*>(L.pool_sb + (size_t)s_idx[k] * L.sb_stride) + (size_t)row * g.gpr,
                 n * ws, m);
    }
  }
  if (lane == 0) S.misc[kBpar] = l & 1;
}

// Phase C's layout in A for the CTA's n output rows: codes of slot k at
// k*n*wqf, scale/bias rows at (K+1)*n*wqf + k*n*wsf, partial results
// ys[k*n + r] after both.
__device__ __forceinline__ size_t c_sb(const FGeo& g, int K, int n, int k) {
  return (size_t)(K + 1) * n * g.wqf + (size_t)k * n * g.wsf;
}
__device__ __forceinline__ size_t c_ys(const FGeo& g, int K, int n) {
  return (size_t)up16((K + 1) * n * (g.wqf + g.wsf));
}

// Warp 14: issue phase C's copies into A: the CTA's rows of the down matrices
// of the K selected experts and of the shared expert; lane k copies slot k's
// codes, lane 16 + k its scale/bias rows.
template <int BITS>
__device__ void issue_C(const FusedParams& P, int l, const FSmem& S) {
  const FGeo& g = P.g;
  const FusedLayer& L = P.layers[l];
  const int f = P.f, K = P.K, lane = threadIdx.x & 31;
  const int cb = S.misc[kCb], n = S.misc[kCe] - cb;
  fence_proxy_async();
  if (lane == 0) mbar_expect_tx(S.mC, (uint32_t)((K + 1) * n * (g.wqf + g.wsf)));
  __syncwarp();
  const int k = lane & 15;
  if (k <= K && n > 0) {
    const uint32_t* q;
    const uint16_t* sb;
    if (k < K) {
      const int e = S.misc[kIdx + k];
      q = L.pool_q + (size_t)e * L.q_stride;
      sb = L.pool_sb + (size_t)e * L.sb_stride;
    } else {
      q = L.shared_q;
      sb = L.shared_sb;
    }
    if (lane < 16)
      bulk_g2s(S.A + (size_t)k * n * g.wqf, q + 2 * (size_t)f * g.wpr + (size_t)cb * (f * BITS / 32),
               (uint32_t)n * g.wqf, S.mC);
    else
      bulk_g2s(S.A + c_sb(g, K, n, k), sb + 2 * (size_t)f * g.gpr * 2 + (size_t)cb * (f / kGroup) * 2,
               (uint32_t)n * g.wsf, S.mC);
  }
  if (lane == 0) S.misc[kCpar] = l & 1;
}

// Phase C's dot products: rows [0, n) of the down matrices of slots 0..K
// (staged SwiGLU outputs of slot k). The (slot, row group) work is cut into
// chunks of at most kCU row groups of one slot (as few chunks per slot as
// that allows, of near-equal size). A warp loads the slot's staged input for
// its part once per chunk, runs the chunk's rows as independent chains and
// reduces them together (with the same addition tree as row_reduce, so the
// results are bit-identical to the batched kernels'); ys[k * n + r] = row r
// of slot k.
constexpr int kCU = 9;

template <int BITS>
__device__ __forceinline__ void down_rows(const unsigned char* Bm, const FGeo& g, int K, int n, const XStage& sth,
                                          const RowGeo& rgf, float* ys, int warp, int lane) {
  using G = Geo<BITS>;
  const int nrg = (n + rgf.RPP - 1) / rgf.RPP;
  const int cpk = (nrg + kCU - 1) / kCU;  // chunks per slot
  const int nch = cpk * (K + 1);
  const int lp = lane % rgf.LPR, rs = lane / rgf.LPR;
  const int rstep = rgf.RPP * g.wqf, sstep = rgf.RPP * g.wsf;
#pragma unroll 1
  for (int c = warp; c < nch; c += kFWarps) {
    const int k = c / cpk, ci = c - k * cpk;
    const int g0 = nrg * ci / cpk, g1 = nrg * (ci + 1) / cpk;  // at most kCU row groups
    uint4 xc[4 * G::kNch];
    uint2 xh[4 * G::kNch];
    load_part_x<BITS>(sth, k, 0, lp, rgf, xc, xh);
    const float2 pi = sth.partinfo[k * rgf.P + lp];
    const int r0 = g0 * rgf.RPP + rs;
    const unsigned char* qb = Bm + (size_t)k * n * g.wqf + (size_t)r0 * g.wqf + lp * 16;
    const unsigned char* sbb = Bm + c_sb(g, K, n, k) + (size_t)r0 * g.wsf + part_group<BITS>(lp) * 4;
    float v[kCU];
#pragma unroll
    for (int u = 0; u < kCU; ++u) {
      v[u] = 0.f;
      if (g0 + u < g1 && r0 + u * rgf.RPP < n) {
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
        if (g0 + u < g1 && rloc < n) ys[k * n + rloc] = y;
      }
#pragma unroll
      for (int u = 8; u < kCU; ++u) {
        const float y2 = row_reduce(v[u], rgf.LPR);
        const int rloc = r0 + u * rgf.RPP;
        if (lp == 0 && g0 + u < g1 && rloc < n) ys[k * n + rloc] = y2;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kCU; ++u) {
        const float y = row_reduce(v[u], rgf.LPR);
        const int rloc = r0 + u * rgf.RPP;
        if (lp == 0 && g0 + u < g1 && rloc < n) ys[k * n + rloc] = y;
      }
    }
  }
}

// SwiGLU outputs read through L2 (written by other SMs during this layer).
struct L2Src {
  const float* x;
  int ld;
  __device__ void load8(int t, int k0, float* v) const {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(x + (size_t)t * ld + k0));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(x + (size_t)t * ld + k0 + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// --------------------------------------------------------------- the kernel
template <int BITS, bool TRACE>
__global__ void __launch_bounds__(kFThreads, 1) k_fused_decode(const __grid_constant__ FusedParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const FGeo& g = P.g;
  const int d = P.d, f = P.f, E = P.E, K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Ctrl* ctrl = P.ctrl;
  const RowGeo rgf = row_geo(f, BITS);

  FSmem S;
  S.mR = reinterpret_cast<uint64_t*>(smem);
  S.mC = S.mR + 1;
  S.mS = S.mR + 2;
  S.mB = S.mS + kMaxSC;
  S.misc = reinterpret_cast<int*>(smem + g.o_misc);
  S.A = smem + g.o_a;
  S.B = smem + g.o_b;
  int* misc = S.misc;
  float* miscf = reinterpret_cast<float*>(misc);
  uint16_t* a_s = reinterpret_cast<uint16_t*>(smem + g.o_as);
  const XStage sta = xstage_carve(smem + g.o_sta, 1, d);
  // This CTA's rows [cb, ce) of the residual stream (stack mode; the input
  // token before layer 0). The CTA writes the same rows every layer, so the
  // combine adds to this copy instead of reading them back from L2.
  float* hres = reinterpret_cast<float*>(smem + g.o_hres);

  if (tid == 0) {
    mbar_init(S.mR, 1);
    mbar_init(S.mC, 1);
    for (int j = 0; j < kMaxSC; ++j) mbar_init(&S.mS[j], 1);
    for (int j = 0; j < kMaxBC; ++j) mbar_init(&S.mB[j], 1);
    misc[kApar] = misc[kSpar] = misc[kBpar] = misc[kCpar] = -1;
    // shared gate/up units of this CTA
    int b, e;
    if (g.s1_nr > 0 && (int)blockIdx.x >= g.nRouter) {
      b = ((int)blockIdx.x - g.nRouter) * g.s1_nr;
      e = b + g.s1_nr;
    } else {
      fsplit(f - g.s1_rest0, blockIdx.x, g.s1_nparts, b, e);
      b += g.s1_rest0;
      e += g.s1_rest0;
    }
    misc[kS1b] = b;
    misc[kS1e] = e;
    misc[kNS] = make_chunks(b, e, f, kMaxSC, misc + kChS);
    fsplit(K * f, blockIdx.x, g.nC, b, e);  // selected gate/up units (unit k*f + row)
    misc[kBb] = b;
    misc[kBe] = e;
    misc[kNB] = make_chunks(b, e, f, kMaxBC, misc + kChB);
    fsplit(d, blockIdx.x, g.nC, b, e);  // output rows
    misc[kCb] = b;
    misc[kCe] = e;
    fence_mbar_init();
  }
  __syncthreads();
  const int cb = misc[kCb], nrows_c = misc[kCe] - cb;
  if (P.stack)
    for (int k = tid; k < nrows_c; k += kFThreads) hres[k] = bf16f(P.x_in[cb + k]);
  if (warp == 0) {
    if (lane == 0) issue_router(P, 0, S);
    issue_shared(P, 0, S);
  }

  for (int l = 0; l < P.n_layers; ++l) {
    const FusedLayer& L = P.layers[l];
    const uint32_t par = (uint32_t)(l & 1);
    const bool has_gate = L.sgate != nullptr;
    stamp<TRACE>(P, l, 0);

    // ---------------- A0: layer input (RMSNorm of the residual in stack mode)
    if (P.stack) {
      // the RMSNorm weight does not depend on the previous layer: load it first
      constexpr int kA0 = 2;  // 8-element slices per thread (d <= 8192)
      uint4 rv[kA0];
#pragma unroll
      for (int i = 0; i < kA0; ++i) {
        const int c = tid + i * kFThreads;
        rv[i] = c < d / 8 ? ldg_stream16(L.rho + 8 * c) : make_uint4(0, 0, 0, 0);
      }
      if (l > 0 && !cta_wait(&ctrl->misc[4], g.nC * l, ctrl, P.timeout_ns, S)) return;
      stamp<TRACE>(P, l, 1);
      float hv[kA0][8];
#pragma unroll
      for (int i = 0; i < kA0; ++i) {
        const int c = tid + i * kFThreads;
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[i][j] = 0.f;
        if (c < d / 8) {
          if (l == 0) {
            unpack_bf16x8(*reinterpret_cast<const uint4*>(P.x_in + 8 * c), hv[i]);
          } else {
            const float4 h0 = __ldcg(reinterpret_cast<const float4*>(P.h + 8 * c));
            const float4 h1 = __ldcg(reinterpret_cast<const float4*>(P.h + 8 * c + 4));
            hv[i][0] = h0.x; hv[i][1] = h0.y; hv[i][2] = h0.z; hv[i][3] = h0.w;
            hv[i][4] = h1.x; hv[i][5] = h1.y; hv[i][6] = h1.z; hv[i][7] = h1.w;
          }
        }
      }
      // sum of squares: the input's own (layer 0), else the previous layer's per-CTA sums, in order
      float ss = 0.f;
      if (l == 0) {
#pragma unroll
        for (int i = 0; i < kA0; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) ss = fmaf(hv[i][j], hv[i][j], ss);
      } else if (warp == 0) {
        const float* part = P.part_ss + (l & 1) * g.nC;
        for (int c0 = 0; c0 < g.nC; c0 += 8 * 32) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = c0 + i * 32 + lane < g.nC ? __ldcg(part + c0 + i * 32 + lane) : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) ss += v[i];
        }
      }
      ss = warp_sum(ss);
      if (l == 0) {  // every warp summed part of the input
        if (lane == 0) miscf[kRed + warp] = ss;
        __syncthreads();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < kFWarps; ++w) s += miscf[kRed + w];
          miscf[kR] = 1.f / sqrtf(s / (float)d + P.eps);
        }
      } else if (tid == 0) {  // warp 0 alone summed the previous layer's per-CTA sums
        miscf[kR] = 1.f / sqrtf(ss / (float)d + P.eps);
      }
      __syncthreads();
      const float r = miscf[kR];
#pragma unroll
      for (int i = 0; i < kA0; ++i) {
        const int c = tid + i * kFThreads;
        if (c < d / 8) {
          float rho[8];
          unpack_bf16x8(rv[i], rho);
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
    stamp<TRACE>(P, l, 2);

    // ---------------- A1: router rows (in B), logits published as tagged words
    {
      const int rloc = warp / g.qr, qtr = warp - rloc * g.qr;
      const int row = (int)blockIdx.x * g.rpc + rloc;
      const bool valid = rloc < g.rpc && row < E + (has_gate ? 1 : 0);
      float v = 0.f;
      if (valid) {
        mbar_wait(S.mR, par, ctrl, P.timeout_ns);
        const int c0 = qtr * (d / g.qr);
        v = router_dot(reinterpret_cast<const uint16_t*>(S.B) + (size_t)rloc * d, a_s, c0, d / g.qr / 256, lane);
      }
      if (lane == 0) miscf[kRed + warp] = v;
      __syncthreads();
      if (valid && qtr == 0 && lane == 0) {
        float s = 0.f;
        for (int q = 0; q < g.qr; ++q) s += miscf[kRed + warp + q];
        st_relaxed_u64(P.ltag + row, ((unsigned long long)(l + 1) << 32) | __float_as_uint(s));
      }
    }
    stamp<TRACE>(P, l, 3);
    // the layer input as 24-bit fixed point for the gate/up rows (its closing
    // barrier also orders the reset of the failure flag before the logits poll)
    if (tid == 0) misc[kFail] = 0;
    stage_x24<BITS>(StridedSrc<uint16_t>{a_s, d}, 1, d, sta);
    stamp<TRACE>(P, l, 12);

    // ---------------- S: selection from the complete logits (every CTA)
    constexpr int kSelMaxK = 8;  // the largest top_k the kernel takes
    // Thread tid polls the tagged words of rows tid, tid + 512 (, tid + 1024)
    // and keeps the logits in registers as order-preserving keys; every warp
    // selects its own top K (larger key first, lower index on equal keys) and
    // warp 0 merges the warps' candidates the same way: the top K of the
    // union lie among every part's top K, so set and order equal a selection
    // over all logits at once (the router kernel's block_topk).
    {
      int* ck = reinterpret_cast<int*>(S.B);  // [16][K] candidate keys (the router rows are done;
      int* ci = ck + kFWarps * kSelMaxK;      // [16][K] their rows       phase B's copies follow)
      const unsigned tag = (unsigned)l + 1u;  // the words are zero when a launch starts
      const int nrows = E + (has_gate ? 1 : 0);
      int key[3];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int row = tid + j * kFThreads;
        key[j] = INT_MIN;
        if (row >= nrows) continue;
        unsigned long long v;
        unsigned long long t0 = 0;
        bool ok = true;
        for (int it = 1; (unsigned)((v = ld_relaxed_u64(P.ltag + row)) >> 32) != tag; ++it) {
          if ((it & 31) == 0) {
            const unsigned long long t = globaltimer();
            if (t0 == 0) t0 = t;
            if (aborted(ctrl) || (long long)(t - t0) > P.timeout_ns || it > (int)kMaxSpin) {
              if (!aborted(ctrl)) raise_timeout(ctrl);
              misc[kFail] = 1;
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        const float f = __uint_as_float((unsigned)v);
        if (row < E)
          key[j] = fkey(f);
        else
          miscf[kL + K] = f;  // the shared-gate logit
      }
#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        const int m = redux_max(max(key[0], max(key[1], key[2])));
        int li = INT_MAX;
#pragma unroll
        for (int j = 2; j >= 0; --j)
          if (key[j] == m) li = tid + j * kFThreads;
        const int bi = redux_min(li);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          if (tid + j * kFThreads == bi) key[j] = INT_MIN;
        if (lane == 0) {
          ck[warp * K + k] = m;
          ci[warp * K + k] = m == INT_MIN ? INT_MAX : bi;
        }
      }
      __syncthreads();
      if (misc[kFail]) {
        if (tid == 0) drain_copies(S);
        return;
      }
      stamp<TRACE>(P, l, 5);
      if (warp == 0) {
        const int n = kFWarps * K;  // <= 128: four per lane
        int kk[4], ii[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = lane + 32 * j;
          kk[j] = c < n ? ck[c] : INT_MIN;
          ii[j] = c < n ? ci[c] : INT_MAX;
        }
        int sel = 0, selk = INT_MIN;
#pragma unroll 1
        for (int k = 0; k < K; ++k) {
          const int m = redux_max(max(max(kk[0], kk[1]), max(kk[2], kk[3])));
          int li = INT_MAX;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (kk[j] == m) li = min(li, ii[j]);
          const int bi = redux_min(li);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (ii[j] == bi) kk[j] = INT_MIN;
          if (lane == k) {
            sel = bi;
            selk = m;
          }
        }
        if (lane < K) {
          misc[kIdx + lane] = sel;
          miscf[kL + lane] = __int_as_float(selk >= 0 ? selk : selk ^ 0x7fffffff);  // the key's logit
        }
        if (lane == 0 && !has_gate) miscf[kL + K] = 0.f;
      }
      __syncthreads();
      stamp<TRACE>(P, l, 11);
    }

    // ---------------- B: the selected experts' gate/up units (in B)
    // Copied in two waves: two thirds of the chunks (rounded up) at once, the
    // rest after the shared units, so that the first wave lands early and its
    // units are computed while the rest streams in (same box, 24-layer 4-bit
    // stack: one wave 20.09, half 19.97, two thirds 19.51, a third 19.98 us
    // per layer).
    const int nB1 = (2 * misc[kNB] + 2) / 3;
    if (warp == kFWarps - 1) {
      issue_B(P, l, S, 0, nB1);  // the last warp: its phase-B units (if any) come last
      if (TRACE && lane == 0 && misc[kNB] > 0) {  // when the first chunk lands
        mbar_wait(&S.mB[0], par, ctrl, P.timeout_ns);
        stamp<TRACE>(P, l, 14);
      }
    }
    if (warp == 0) {  // the routing weights (used by the combine) while the copies start
      block_topk_weights(miscf + kL, K, has_gate, miscf + kW);
      __syncwarp();
      if (blockIdx.x == 0 && lane < K) {
        if (P.idx_out) P.idx_out[l * K + lane] = misc[kIdx + lane];
        if (P.w_out) P.w_out[l * K + lane] = miscf[kW + lane];
      }
      if (blockIdx.x == 0 && lane == 0 && P.gamma_out) P.gamma_out[l] = miscf[kW + K];
    }
    // The shared expert's gate/up units (copied into A during the previous
    // layer) do not gate the selection, so they run here, while phase B's
    // rows stream in; then A takes the down rows, which land behind them.
    run_units<BITS>(S.A, misc[kS1b], misc[kS1e], misc + kChS, misc[kNS], S.mS, par, ctrl, P.timeout_ns, sta, g,
                    P.hk + (size_t)K * f + misc[kS1b], kFWarps - 1 - warp, lane);
    __syncthreads();
    stamp<TRACE>(P, l, 4);
    if (warp == kFWarps - 2) {
      issue_B(P, l, S, nB1, misc[kNB]);
      issue_C<BITS>(P, l, S);
    }
    if (TRACE && warp == kFWarps - 1 && lane == 0 && misc[kNB] > 0) {  // when the last chunk lands
      mbar_wait(&S.mB[misc[kNB] - 1], par, ctrl, P.timeout_ns);
      stamp<TRACE>(P, l, 15);
    }
    run_units<BITS>(S.B, misc[kBb], misc[kBe], misc + kChB, misc[kNB], S.mB, par, ctrl, P.timeout_ns, sta, g,
                    P.hk + misc[kBb], warp, lane);  // unit k*f + row
    stamp<TRACE>(P, l, 6);
    cta_arrive(&ctrl->misc[3]);

    // ---------------- C: down rows + combine (+ residual)
    if (!cta_wait(&ctrl->misc[3], g.nC * (l + 1), ctrl, P.timeout_ns, S)) return;
    stamp<TRACE>(P, l, 7);
    // the next layer's router rows (needed first; its shared units follow the down rows)
    if (tid == 0 && l + 1 < P.n_layers) issue_router(P, l + 1, S);
    // every SwiGLU output, straight from L2 into the staged format
    const XStage sth = xstage_carve(S.B + up16(g.rpc * 2 * d), K + 1, f);  // after the next layer's router rows
    stage_x24_pairs<BITS>(L2Src{P.hk, f}, K + 1, f, sth);
    stamp<TRACE>(P, l, 13);
    mbar_wait(S.mC, par, ctrl, P.timeout_ns);
    stamp<TRACE>(P, l, 9);
    float* ys = reinterpret_cast<float*>(S.A + c_ys(g, K, nrows_c));
    down_rows<BITS>(S.A, g, K, nrows_c, sth, rgf, ys, warp, lane);
    __syncthreads();
    stamp<TRACE>(P, l, 10);
    // combine in fixed order: routed experts k = 0..K-1, then the shared expert (k = K)
    float ss = 0.f;
    for (int rl = tid; rl < nrows_c; rl += kFThreads) {
      const int row = cb + rl;
      float o = 0.f;
      for (int k = 0; k <= K; ++k) o = fmaf(miscf[kW + k], ys[k * nrows_c + rl], o);
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
    if (P.stack) {
      ss = warp_sum(ss);
      if (lane == 0) miscf[kRed + warp] = ss;
      __syncthreads();
      if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < kFWarps; ++w) s += miscf[kRed + w];
        P.part_ss[((l + 1) & 1) * g.nC + blockIdx.x] = s;
      }
    }
    // A is free again (down rows and partial results consumed): the next
    // layer's shared gate/up rows
    __syncthreads();
    if (warp == 0 && l + 1 < P.n_layers) issue_shared(P, l + 1, S);
    stamp<TRACE>(P, l, 8);
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
      if (lane == 0) miscf[kR] = 1.f / sqrtf(s / (float)d + P.eps);
    }
    __syncthreads();
    const float r = miscf[kR];
    for (int k = tid; k < nrows_c; k += kFThreads) {
      const float hv = hres[k];  // written by this thread in the last layer's combine
      if (P.x_next) P.x_next[cb + k] = f2bf(hv * r);
      if (P.h_out) P.h_out[cb + k] = hv;
    }
  }
  // the last CTA out resets the counters and clears the tagged logits for the
  // next launch (every other CTA has read them by now)
  __syncthreads();
  if (tid == 0) misc[kLast] = atomicAdd(&ctrl->misc[5], 1) == g.nC - 1;
  __syncthreads();
  if (misc[kLast]) {
    for (int e = tid; e <= E; e += kFThreads) P.ltag[e] = 0ull;
    if (tid == 0) {
      for (int i = 1; i <= 5; ++i) ctrl->misc[i] = 0;
      __threadfence();
    }
  }
}

// --------------------------------------------------------------- wait self-test
// Two CTAs wait on a counter nothing increments, with a short limit: the
// bounded wait must give up, write BGQ_ERR_TIMEOUT and return. Exercises the
// same grid-wide wait the decode kernel uses, without faulting anything.
__global__ void k_wait_selftest(Ctrl* ctrl, long long timeout_ns) {
  __shared__ int misc[kMiscInts];
  FSmem S{};
  S.misc = misc;
  if (threadIdx.x == 0) {
    misc[kApar] = misc[kSpar] = misc[kBpar] = misc[kCpar] = -1;
    misc[kNS] = misc[kNB] = 0;
  }
  __syncthreads();
  if (!cta_wait(&ctrl->misc[6], 1 << 30, ctrl, timeout_ns, S)) return;
  if (threadIdx.x == 0) atomicExch(&ctrl->status, BGQ_OK);  // not reached: nothing sets misc[6]
}

cudaError_t launch_wait_selftest(Ctrl* ctrl, long long timeout_ns, cudaStream_t s) {
  k_wait_selftest<<<2, 64, 0, s>>>(ctrl, timeout_ns);
  return cudaGetLastError();
}

// --------------------------------------------------------------- host side
size_t fused_smem_bytes(int d, int f, int K, int bits) {
  return (size_t)fused_geo(num_sms(), d, f, 1024, K, bits).total;
}

bool fused_supported(int d, int f, int E, int K, int bits) {
  if (K < 1 || K > 8 || E < K || E > 1024) return false;
  if (d % 256 || f % 256) return false;  // scale/bias rows of 16-byte multiples (bulk copies)
  if (d > 2048 && d % 1024) return false;  // router slices of 1024 columns, or one slice of <= 2048
  if (d > 8192) return false;              // two 8-element slices per thread in the RMSNorm
  const int Pd = d * bits / 128, Pf = f * bits / 128;
  if (Pd < 32 || Pd % 32 || Pd / 32 > 4) return false;  // d-rows: all lanes, <= 4 parts each
  if (Pf < 1 || Pf > 32 || 32 % Pf) return false;       // f-rows: one part per lane
  const int nC = num_sms();
  const FGeo g = fused_geo(nC, d, f, E, K, bits);
  if (g.nRouter > nC) return false;  // every router row owned by one CTA
  if (g.nBmax > kMaxB) return false;
  // bulk-copy chunks per CTA (the kernel's make_chunks)
  auto chunks = [&](int b, int e) {
    int n = 0;
    for (int start = b; start < e; ++n) {
      int lim = start + kCH < e ? start + kCH : e;
      const int seg = (start / f + 1) * f;
      start = seg < lim ? seg : lim;
    }
    return n;
  };
  for (int c = 0; c < nC; ++c) {
    int b, e;
    fsplit(K * f, c, nC, b, e);
    if (chunks(b, e) > kMaxBC) return false;
    if (c >= g.nRouter && g.s1_nr > 0) {
      b = (c - g.nRouter) * g.s1_nr;
      e = b + g.s1_nr;
    } else {
      fsplit(f - g.s1_rest0, c, g.s1_nparts, b, e);
      b += g.s1_rest0;
      e += g.s1_rest0;
    }
    if (e - b > kMaxS1 || chunks(b, e) > kMaxSC) return false;
  }
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  return (size_t)g.total + 1024 <= (size_t)optin;
}

cudaError_t launch_fused(const FusedParams& P0, int bits, cudaStream_t s) {
  const int nC = num_sms();
  FusedParams P = P0;
  P.g = fused_geo(nC, P.d, P.f, P.E, P.K, bits);
  const size_t sm = (size_t)P.g.total;
  void* kern = P.trace ? (bits == 4 ? (void*)k_fused_decode<4, true> : (void*)k_fused_decode<2, true>)
                       : (bits == 4 ? (void*)k_fused_decode<4, false> : (void*)k_fused_decode<2, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&P};
  return cudaLaunchCooperativeKernel(kern, dim3(nC), dim3(kFThreads), args, sm, s);
}

}  // namespace bgq
