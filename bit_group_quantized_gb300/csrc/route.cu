// route.cu — fused router GEMV + softmax + top-K + renormalise (+ grouping plan).
//
// Flash-MoE page, section "架构设计：SSD当显存用": after the routing logits are
// computed, softmax and top-K select the experts (K = 4 of 512 per section
// "先搞清楚为什么这件事很难"). The page runs softmax + topK on the CPU; here it
// is the tail of the router kernel: every CTA computes a slice of the logits,
// and the last CTA to finish (atomic counter, no waiting) selects the experts.
//
//   l[e] = router[e] . x (fp32), top-K by logit, ties to the lower index,
//   largest first, w_k = p[idx_k] / sum_j p[idx_j] with p = softmax(l), which
//   is computed as exp(l_k - l_max) / sum_j exp(l_j - l_max) over the selected
//   logits (the full softmax denominator cancels),
//   gamma = sigmoid(shared_gate . x).
//
// With a plan pointer, the last CTA also groups the (token, slot) pairs by
// expert (counting sort, stable by token then slot) into grouped-GEMV tasks of
// at most 8 tokens, routed experts in ascending order, then the shared expert.
#include "../../include/bgq.h"
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace bgq {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = 8;
constexpr int kRouteTok = 8;       // tokens per x chunk in shared memory
constexpr int kRouteMaxVec = 8;    // 16-byte weight vectors per lane held in registers
constexpr int kMaxExperts = 1024;  // top-K registers: 32 logits per lane
constexpr int kMaxTopK = 8;

struct RouteGeo {
  int sk;        // warps per row (split-K)
  int rows_cta;  // rows per CTA
  int nvec;      // 16-byte vectors per lane per row slice
};
// Rows are cut into slices of 1024 columns when d is a multiple of 1024 (the
// same cut as the persistent batch-1 kernel, so both sum a logit in the same
// order and give bit-identical results), else one slice per row.
__host__ __device__ inline RouteGeo route_geo(int d) {
  RouteGeo g;
  g.sk = (d >= 1024 && d % 1024 == 0) ? d / 1024 : 1;
  g.rows_cta = kRouteWarps / g.sk;
  g.nvec = d / g.sk / 256;
  return g;
}
bool route_shape_ok(int d) {
  if (d <= 0 || d % 256) return false;
  RouteGeo g = route_geo(d);
  return g.sk <= kRouteWarps && d % (256 * g.sk) == 0 && g.nvec <= kRouteMaxVec;
}

__device__ void topk_one_token(const float* __restrict__ lg, int E, int K, float zgate, bool has_gate, int t,
                               int32_t* idx, float* w, float* gamma, float* logits_out, int* sel_out) {
  const int lane = threadIdx.x & 31;
  float v[kMaxExperts / 32];
  const int per = (E + 31) / 32;
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    int e = i * 32 + lane;
    v[i] = (i < per && e < E) ? __ldcg(lg + e) : -INFINITY;
    if (logits_out && i < per && e < E) logits_out[(size_t)t * E + e] = v[i];
  }
  // K rounds of arg-max; (value, index) order: larger value, then lower index.
  unsigned taken = 0u;
  int sel[kMaxTopK];
  float selv[kMaxTopK];
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      int e = i * 32 + lane;
      bool ok = i < per && e < E && !((taken >> i) & 1u);
      if (ok && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(kFull, bv, o);
      int oi = __shfl_xor_sync(kFull, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    sel[k] = bi;
    selv[k] = bv;
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
  }
  if (lane == 0) {
    // softmax over all E followed by renormalisation over the K selected is a
    // softmax over the selected logits (the full denominator cancels); selv[0]
    // is the largest logit.
    float p[kMaxTopK], ps = 0.f;
    for (int k = 0; k < K; ++k) {
      p[k] = expf(selv[k] - selv[0]);
      ps += p[k];
    }
    for (int k = 0; k < K; ++k) {
      idx[t * K + k] = sel[k];
      w[t * K + k] = p[k] / ps;
      if (sel_out) sel_out[t * K + k] = sel[k];
    }
    if (gamma) gamma[t] = has_gate ? 1.f / (1.f + expf(-zgate)) : 1.f;
  }
}

// Block-wide exclusive scan of three int arrays a0, a1, a2 of n entries in
// shared memory, in place, in one pass (each thread takes a contiguous run of
// ceil(n / blockDim) entries); the three totals go to tot[0..2]. wt: 96 ints.
__device__ void block_exclusive_scan3(int* a0, int* a1, int* a2, int n, int* wt, int* tot) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per;
  int l0 = 0, l1 = 0, l2 = 0;
  for (int i = 0; i < per; ++i)
    if (lo + i < n) {
      l0 += a0[lo + i];
      l1 += a1[lo + i];
      l2 += a2[lo + i];
    }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int c0 = l0, c1 = l1, c2 = l2;  // inclusive within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v0 = __shfl_up_sync(kFull, c0, o), v1 = __shfl_up_sync(kFull, c1, o), v2 = __shfl_up_sync(kFull, c2, o);
    if (lane >= o) {
      c0 += v0;
      c1 += v1;
      c2 += v2;
    }
  }
  if (lane == 31) {
    wt[warp] = c0;
    wt[32 + warp] = c1;
    wt[64 + warp] = c2;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warp totals
    const int t0 = lane < nw ? wt[lane] : 0, t1 = lane < nw ? wt[32 + lane] : 0, t2 = lane < nw ? wt[64 + lane] : 0;
    int i0 = t0, i1 = t1, i2 = t2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v0 = __shfl_up_sync(kFull, i0, o), v1 = __shfl_up_sync(kFull, i1, o), v2 = __shfl_up_sync(kFull, i2, o);
      if (lane >= o) {
        i0 += v0;
        i1 += v1;
        i2 += v2;
      }
    }
    wt[lane] = i0 - t0;
    wt[32 + lane] = i1 - t1;
    wt[64 + lane] = i2 - t2;
    if (lane == 31) {
      tot[0] = i0;
      tot[1] = i1;
      tot[2] = i2;
    }
  }
  __syncthreads();
  int r0 = wt[warp] + c0 - l0, r1 = wt[32 + warp] + c1 - l1, r2 = wt[64 + warp] + c2 - l2;
  for (int i = 0; i < per; ++i)
    if (lo + i < n) {
      const int v0 = a0[lo + i], v1 = a1[lo + i], v2 = a2[lo + i];
      a0[lo + i] = r0;
      a1[lo + i] = r1;
      a2[lo + i] = r2;
      r0 += v0;
      r1 += v1;
      r2 += v2;
    }
  __syncthreads();
}

// Shared-memory ints build_plan needs for B tokens, top-K and E experts.
__host__ __device__ inline int plan_scratch_ints(int B, int K, int E) { return 4 * E + 104 + B * K; }

// The grouping plan from the selections sel[B*K] (token-major): routed
// experts with fewer than big_min tokens become grouped-GEMV tasks of at most
// kTaskTok tokens (stable: token order, then slot), the others tensor-core
// tasks; then the shared expert (every token, slot K). `s_cnt`:
// plan_scratch_ints(B, K, E) ints of shared memory.
__device__ void build_plan(const int* sel, int B, int K, int E, int big_min, Plan* plan, int* s_cnt) {
  const int npairs = B * K;
  Task* tasks = plan_tasks(plan);
  BigTask* big = plan_big(plan, B, K);
  int* ptok = plan_ptok(plan, B, K);
  int* pslot = plan_pslot(plan, B, K);
  int* s_first = s_cnt + E;       // task index of each small expert's first chunk
  int* s_pfirst = s_cnt + 2 * E;  // pair offset of each big expert
  int* s_bidx = s_cnt + 3 * E;    // big-task index of each big expert
  int* wt = s_cnt + 4 * E;        // [96] scan scratch, then [3] totals
  int* s_sel = wt + 104;          // [npairs] the selections, staged once
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) s_sel[i] = __ldcg(sel + i);
  __syncthreads();
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) atomicAdd(&s_cnt[s_sel[i]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = s_cnt[e];
    const bool bigc = c >= big_min;
    s_first[e] = bigc ? 0 : (c + kTaskTok - 1) / kTaskTok;
    s_pfirst[e] = bigc ? c : 0;
    s_bidx[e] = bigc ? 1 : 0;
  }
  __syncthreads();
  block_exclusive_scan3(s_first, s_pfirst, s_bidx, E, wt, wt + 96);
  const int nsmall = wt[96], nbigpairs = wt[97], nbigr = wt[98];
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    const int e = s_sel[i];
    int r = 0;  // earlier pairs of the same expert
    for (int j = 0; j < i; ++j) r += (s_sel[j] == e);
    if (s_cnt[e] >= big_min) {
      ptok[s_pfirst[e] + r] = i / K;
      pslot[s_pfirst[e] + r] = i % K;
      if (r == 0) big[s_bidx[e]] = BigTask{e, s_cnt[e], s_pfirst[e], 0};
    } else {
      Task& tk = tasks[s_first[e] + r / kTaskTok];
      const int pos = r % kTaskTok;
      tk.tok[pos] = i / K;
      tk.slot[pos] = i % K;
      if (pos == 0) {
        tk.expert = e;
        const int left = s_cnt[e] - (r / kTaskTok) * kTaskTok;
        tk.ntok = left < kTaskTok ? left : kTaskTok;
      }
    }
  }
  // the shared expert takes every token (slot K)
  int nshared = 0, nbig = nbigr;
  if (B >= big_min) {
    for (int t = threadIdx.x; t < B; t += blockDim.x) {
      ptok[nbigpairs + t] = t;
      pslot[nbigpairs + t] = K;
    }
    if (threadIdx.x == 0) big[nbigr] = BigTask{-1, B, nbigpairs, 0};
    nbig = nbigr + 1;
  } else {
    nshared = (B + kTaskTok - 1) / kTaskTok;
    for (int c = threadIdx.x; c < nshared; c += blockDim.x) {
      Task& tk = tasks[nsmall + c];
      tk.expert = -1;
      const int n = B - c * kTaskTok;
      tk.ntok = n < kTaskTok ? n : kTaskTok;
      for (int i = 0; i < tk.ntok; ++i) {
        tk.tok[i] = c * kTaskTok + i;
        tk.slot[i] = K;
      }
    }
  }
  if (threadIdx.x == 0) {
    plan->ntasks = nsmall + nshared;
    plan->nbig = nbig;
  }
  // each tensor-core task's first row in the staged activations: the sum of
  // the earlier tasks' token counts rounded up to 16
  __syncthreads();
  if (threadIdx.x == 0) {
    int rows = 0;
    for (int t = 0; t < nbig; ++t) {
      big[t].pad = rows;
      rows += (big[t].ntok + 15) & ~15;
    }
  }
}

__global__ void __launch_bounds__(kRouteThreads)
k_route(const uint16_t* __restrict__ router, const uint16_t* __restrict__ sgate, const uint16_t* __restrict__ x, int B,
        int d, int E, int K, float* __restrict__ lg, Ctrl* ctrl, int32_t* __restrict__ idx, float* __restrict__ w,
        float* __restrict__ gamma, float* __restrict__ logits_out, Plan* plan, int big_min, int* __restrict__ sel_ws) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                       // [kRouteTok][d]
  float* red = reinterpret_cast<float*>(smem + (size_t)kRouteTok * d * 2);  // [warps][kRouteTok]
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RouteGeo g = route_geo(d);
  const int nrows = E + (sgate ? 1 : 0);
  const int rloc = warp / g.sk, half = warp - rloc * g.sk;
  const int row = blockIdx.x * g.rows_cta + rloc;
  const bool valid = rloc < g.rows_cta && row < nrows;
  const uint16_t* wrow = (row < E) ? router + (size_t)row * d : sgate;
  const int c0 = half * (d / g.sk);

  uint4 wv[kRouteMaxVec];
#pragma unroll
  for (int i = 0; i < kRouteMaxVec; ++i)
    wv[i] = (valid && i < g.nvec) ? ldg_stream16(wrow + c0 + (i * 32 + lane) * 8) : make_uint4(0, 0, 0, 0);

  for (int t0 = 0; t0 < B; t0 += kRouteTok) {
    const int T = B - t0 < kRouteTok ? B - t0 : kRouteTok;
    __syncthreads();
    for (int i = threadIdx.x; i < T * d / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(x + (size_t)t0 * d)[i];
    __syncthreads();
    float acc[kRouteTok];
#pragma unroll
    for (int t = 0; t < kRouteTok; ++t) acc[t] = 0.f;
#pragma unroll
    for (int i = 0; i < kRouteMaxVec; ++i) {
      if (i < g.nvec) {
        const float wf[8] = {bf16lo(wv[i].x), bf16hi(wv[i].x), bf16lo(wv[i].y), bf16hi(wv[i].y),
                             bf16lo(wv[i].z), bf16hi(wv[i].z), bf16lo(wv[i].w), bf16hi(wv[i].w)};
        const int col = c0 + (i * 32 + lane) * 8;
#pragma unroll
        for (int t = 0; t < kRouteTok; ++t) {
          if (t < T) {
            uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)t * d + col);
            float a = acc[t];
            a = fmaf(wf[0], bf16lo(xv.x), a);
            a = fmaf(wf[1], bf16hi(xv.x), a);
            a = fmaf(wf[2], bf16lo(xv.y), a);
            a = fmaf(wf[3], bf16hi(xv.y), a);
            a = fmaf(wf[4], bf16lo(xv.z), a);
            a = fmaf(wf[5], bf16hi(xv.z), a);
            a = fmaf(wf[6], bf16lo(xv.w), a);
            a = fmaf(wf[7], bf16hi(xv.w), a);
            acc[t] = a;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kRouteTok; ++t) {
      float v = warp_sum(acc[t]);
      if (lane == 0) red[warp * kRouteTok + t] = v;
    }
    __syncthreads();
    if (valid && half == 0 && lane < T) {
      float v = 0.f;
      for (int h = 0; h < g.sk; ++h) v += red[(rloc * g.sk + h) * kRouteTok + lane];
      lg[(size_t)(t0 + lane) * (E + 1) + row] = v;
    }
  }
  // last CTA selects the experts
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int prev = atomicAdd(&ctrl->route_counter, 1);
    s_last = (prev == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = warp; t < B; t += kRouteWarps) {
    float z = sgate ? __ldcg(lg + (size_t)t * (E + 1) + E) : 0.f;
    topk_one_token(lg + (size_t)t * (E + 1), E, K, z, sgate != nullptr, t, idx, w, gamma, logits_out, sel_ws);
  }
  if (plan) {
    __syncthreads();
    __threadfence_block();
    int* s_cnt = reinterpret_cast<int*>(smem);  // reuse: plan_scratch_ints(B, K, E) ints
    build_plan(sel_ws, B, K, E, big_min, plan, s_cnt);
  }
  if (threadIdx.x == 0) ctrl->route_counter = 0;  // ready for the next launch
}

// ---------------------------------------------------------------------------
// Cooperative router: one 512-thread CTA per SM.
//   1. CTA c computes the logits of its share of the rows for every token
//      (rows in 1024-column slices, summed in the same order as above and as
//      the persistent batch-1 kernel, so the logits are bit-identical);
//   2. after a grid-wide counter, CTA t selects token t's experts with the
//      block top-K of the persistent kernel (tokens in parallel instead of
//      one warp each in the last CTA);
//   3. the last CTA to finish step 2 builds the grouping plan.
// The counter wait is bounded like every wait in the library.
// ---------------------------------------------------------------------------
constexpr int kRcThreads = 512;
constexpr int kRcWarps = kRcThreads / 32;
static_assert(kRcWarps == kTopkWarps, "block top-K needs 16 warps");
constexpr long long kRcTimeoutNs = 2000000000ll;

__device__ __forceinline__ unsigned long long rc_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Block barrier, then thread 0 adds 1 to *cnt (release) and waits (acquire)
// until it reaches target. False for the whole block on abort or timeout
// (a timeout writes BGQ_ERR_TIMEOUT and raises the abort flag).
__device__ bool rc_grid_sync(int* cnt, int target, Ctrl* ctrl) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
    int ok = 1;
    const unsigned long long t0 = rc_now();
    long long it = 0;
    while (true) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= target) break;
      if (*(volatile int*)&ctrl->misc[0]) {
        ok = 0;
        break;
      }
      if (++it > (1ll << 26) || (long long)(rc_now() - t0) > kRcTimeoutNs) {
        atomicExch(&ctrl->status, BGQ_ERR_TIMEOUT);
        atomicExch(&ctrl->misc[0], 1);
        ok = 0;
        break;
      }
      if (it > 16) __nanosleep(32);
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__global__ void __launch_bounds__(kRcThreads, 1)
k_route_coop(const uint16_t* __restrict__ router, const uint16_t* __restrict__ sgate, const uint16_t* __restrict__ x,
             int B, int d, int E, int K, float* __restrict__ lg, Ctrl* ctrl, int32_t* __restrict__ idx,
             float* __restrict__ w, float* __restrict__ gamma, float* __restrict__ logits_out, Plan* plan,
             int big_min, int* __restrict__ sel_ws) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                       // [kRouteTok][d]
  float* red = reinterpret_cast<float*>(smem + (size_t)kRouteTok * d * 2);  // [warps][kRouteTok]
  __shared__ int s_idx[kMaxTopK];
  __shared__ float s_w[kMaxTopK + 1];
  __shared__ float s_l[kMaxTopK + 1];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RouteGeo g = route_geo(d);
  const int nrows = E + (sgate ? 1 : 0);
  const int rpp = kRcWarps / g.sk;  // rows per pass
  const int r0 = (int)((long long)nrows * blockIdx.x / gridDim.x);
  const int r1 = (int)((long long)nrows * (blockIdx.x + 1) / gridDim.x);

  // 1. logits of rows [r0, r1) for every token
  for (int rb = r0; rb < r1; rb += rpp) {
    const int rloc = warp / g.sk, half = warp - rloc * g.sk;
    const int row = rb + rloc;
    const bool valid = rloc < rpp && row < r1;
    const uint16_t* wrow = (row < E) ? router + (size_t)row * d : sgate;
    const int c0 = half * (d / g.sk);
    uint4 wv[kRouteMaxVec];
#pragma unroll
    for (int i = 0; i < kRouteMaxVec; ++i)
      wv[i] = (valid && i < g.nvec) ? ldg_stream16(wrow + c0 + (i * 32 + lane) * 8) : make_uint4(0, 0, 0, 0);
    for (int t0 = 0; t0 < B; t0 += kRouteTok) {
      const int T = B - t0 < kRouteTok ? B - t0 : kRouteTok;
      __syncthreads();
      for (int i = threadIdx.x; i < T * d / 8; i += blockDim.x)
        reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(x + (size_t)t0 * d)[i];
      __syncthreads();
      float acc[kRouteTok];
#pragma unroll
      for (int t = 0; t < kRouteTok; ++t) acc[t] = 0.f;
#pragma unroll
      for (int i = 0; i < kRouteMaxVec; ++i) {
        if (i < g.nvec) {
          const float wf[8] = {bf16lo(wv[i].x), bf16hi(wv[i].x), bf16lo(wv[i].y), bf16hi(wv[i].y),
                               bf16lo(wv[i].z), bf16hi(wv[i].z), bf16lo(wv[i].w), bf16hi(wv[i].w)};
          const int col = c0 + (i * 32 + lane) * 8;
#pragma unroll
          for (int t = 0; t < kRouteTok; ++t) {
            if (t < T) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)t * d + col);
              float a = acc[t];
              a = fmaf(wf[0], bf16lo(xv.x), a);
              a = fmaf(wf[1], bf16hi(xv.x), a);
              a = fmaf(wf[2], bf16lo(xv.y), a);
              a = fmaf(wf[3], bf16hi(xv.y), a);
              a = fmaf(wf[4], bf16lo(xv.z), a);
              a = fmaf(wf[5], bf16hi(xv.z), a);
              a = fmaf(wf[6], bf16lo(xv.w), a);
              a = fmaf(wf[7], bf16hi(xv.w), a);
              acc[t] = a;
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kRouteTok; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) red[warp * kRouteTok + t] = v;
      }
      __syncthreads();
      if (valid && half == 0 && lane < T) {
        float v = 0.f;
        for (int h = 0; h < g.sk; ++h) v += red[(rloc * g.sk + h) * kRouteTok + lane];
        lg[(size_t)(t0 + lane) * (E + 1) + row] = v;
      }
    }
  }
  if (!rc_grid_sync(&ctrl->misc[10], (int)gridDim.x, ctrl)) return;

  // 2. token t's experts, tokens spread over the CTAs
  float* lgs = reinterpret_cast<float*>(smem);  // E + 1 logits, then the candidates
  for (int t = blockIdx.x; t < B; t += gridDim.x) {
    __syncthreads();
    for (int e = threadIdx.x; e < nrows; e += blockDim.x) {
      const float v = __ldcg(lg + (size_t)t * (E + 1) + e);
      lgs[e] = v;
      if (logits_out && e < E) logits_out[(size_t)t * E + e] = v;
    }
    __syncthreads();
    block_topk(lgs, reinterpret_cast<int*>(lgs + ((E + 4) & ~3)), E, K, sgate != nullptr, s_idx, s_l, s_w);
    if (threadIdx.x < K) {
      idx[t * K + threadIdx.x] = s_idx[threadIdx.x];
      w[t * K + threadIdx.x] = s_w[threadIdx.x];
      sel_ws[t * K + threadIdx.x] = s_idx[threadIdx.x];
    }
    if (threadIdx.x == 0 && gamma) gamma[t] = s_w[K];
  }

  // 3. the last CTA out builds the plan and resets the counters
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&ctrl->misc[11], 1);
    s_last = prev == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  pdl_trigger();  // every other CTA has left: the grouped kernel behind may take their SMs and wait there
  if (plan) {
    int* s_cnt = reinterpret_cast<int*>(smem);  // plan_scratch_ints(B, K, E) ints
    build_plan(sel_ws, B, K, E, big_min, plan, s_cnt);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ctrl->misc[10] = 0;
    ctrl->misc[11] = 0;
    __threadfence();
  }
}

static size_t route_coop_smem(int d, int E, int B, int K) {
  size_t sm = (size_t)kRouteTok * d * 2 + kRcWarps * kRouteTok * sizeof(float);
  const size_t sm_topk = ((size_t)((E + 4) & ~3) + topk_scratch_ints(E)) * sizeof(float);
  const size_t sm_plan = (size_t)plan_scratch_ints(B, K, E) * sizeof(int);
  if (sm_topk > sm) sm = sm_topk;
  if (sm_plan > sm) sm = sm_plan;
  return sm;
}

cudaError_t launch_route(const uint16_t* router, const uint16_t* sgate, const uint16_t* x, int batch, int d, int E,
                         int K, float* logits_ws, Ctrl* ctrl, int32_t* idx, float* w, float* gamma,
                         float* logits_out, Plan* plan, int big_min, cudaStream_t s) {
  // selected experts scratch for the plan: right after the logits
  int* sel = reinterpret_cast<int*>(logits_ws + (size_t)batch * (E + 1));
  if (E <= kTopkWarps * 64) {
    const size_t smc = route_coop_smem(d, E, batch, K);
    cudaError_t e = cudaFuncSetAttribute(k_route_coop, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smc);
    int per_sm = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_route_coop, kRcThreads, smc);
    if (e != cudaSuccess) return e;
    if (per_sm >= 1) {
      void* args[] = {(void*)&router, (void*)&sgate, (void*)&x,     (void*)&batch, (void*)&d,
                      (void*)&E,      (void*)&K,     (void*)&logits_ws, (void*)&ctrl, (void*)&idx,
                      (void*)&w,      (void*)&gamma, (void*)&logits_out, (void*)&plan, (void*)&big_min, (void*)&sel};
      return cudaLaunchCooperativeKernel((void*)k_route_coop, dim3(num_sms()), dim3(kRcThreads), args, smc, s);
    }
  }
  RouteGeo g = route_geo(d);
  int nrows = E + (sgate ? 1 : 0);
  int grid = (nrows + g.rows_cta - 1) / g.rows_cta;
  size_t sm = (size_t)kRouteTok * d * 2 + kRouteWarps * kRouteTok * sizeof(float);
  size_t sm_plan = (size_t)plan_scratch_ints(batch, K, E) * sizeof(int);
  if (sm_plan > sm) sm = sm_plan;
  if (sm > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  k_route<<<grid, kRouteThreads, sm, s>>>(router, sgate, x, batch, d, E, K, logits_ws, ctrl, idx, w, gamma,
                                          logits_out, plan, big_min, sel);
  return cudaGetLastError();
}

// Plan of one explicit expert over B tokens (slot 0): one tensor-core task for
// B >= big_min, else grouped-GEMV tasks of up to 8 tokens. Plan sized for (B, 0).
__global__ void k_plan_single(Plan* plan, int B, int big_min) {
  pdl_wait();  // an earlier kernel may still read the plan
  pdl_trigger();
  if (B >= big_min) {
    BigTask* big = plan_big(plan, B, 0);
    int* ptok = plan_ptok(plan, B, 0);
    int* pslot = plan_pslot(plan, B, 0);
    for (int t = threadIdx.x; t < B; t += blockDim.x) {
      ptok[t] = t;
      pslot[t] = 0;
    }
    if (threadIdx.x == 0) {
      big[0] = BigTask{-1, B, 0, 0};
      plan->nbig = 1;
      plan->ntasks = 0;
    }
    return;
  }
  const int n = (B + kTaskTok - 1) / kTaskTok;
  for (int c = threadIdx.x; c < n; c += blockDim.x) {
    Task& tk = plan_tasks(plan)[c];
    tk.expert = -1;
    int m = B - c * kTaskTok;
    tk.ntok = m < kTaskTok ? m : kTaskTok;
    for (int i = 0; i < tk.ntok; ++i) {
      tk.tok[i] = c * kTaskTok + i;
      tk.slot[i] = 0;
    }
  }
  if (threadIdx.x == 0) {
    plan->ntasks = n;
    plan->nbig = 0;
  }
}

cudaError_t launch_plan_single(Plan* plan, int batch, int big_min, cudaStream_t s) {
  return launch_overlapped(k_plan_single, 1, 64, 0, s, plan, batch, big_min);
}

}  // namespace bgq
