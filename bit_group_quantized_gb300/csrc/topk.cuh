// topk.cuh — block-wide top-K selection of one token's routing logits.
//
// Flash-MoE page, section "架构设计：SSD当显存用": softmax + top-K pick the
// experts of a token from its routing logits, then the K weights are
// renormalised. Used by the persistent batch-1 kernel and the cooperative
// router kernel (512-thread blocks, 16 warps).
#pragma once

#include <climits>

#include "common.cuh"

namespace bgq {

constexpr int kTopkWarps = 16;  // the block has 16 warps

// Order-preserving map of a float to a signed int (larger float, larger int).
__device__ __forceinline__ int fkey(float v) {
  const int i = __float_as_int(v == 0.f ? 0.f : v);  // -0 and +0 compare equal
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ int redux_max(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ int redux_min(int v) {
  int r;
  asm volatile("redux.sync.min.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Warp-wide selection among n > 32 candidates (keys ck, indices ci in shared
// memory): K rounds of max, lowest index among equal keys, remove. Lane k
// returns the k-th selected index. Rare (ties over many logits), so it is
// kept out of line.
static __device__ __noinline__ int topk_many_candidates(int* ck, const int* ci, int n, int K, int lane) {
  int sel = 0;
  for (int k = 0; k < K; ++k) {
    int lb = INT_MIN;
    for (int c = lane; c < n; c += 32) lb = max(lb, ck[c]);
    const int best = redux_max(lb);
    int li = INT_MAX;
    for (int c = lane; c < n; c += 32)
      if (ck[c] == best) li = min(li, ci[c]);
    const int bi = redux_min(li);
    for (int c = lane; c < n; c += 32)
      if (ci[c] == bi) ck[c] = INT_MIN;
    __syncwarp();
    if (lane == k) sel = bi;
  }
  return sel;
}

// Scratch ints block_topk_select needs for E logits.
__host__ __device__ constexpr int topk_scratch_ints(int E) { return 32 + 2 * E; }

// Top-K selection, run by every CTA on the logits in shared memory (lg[0..E),
// lg[E] = shared-gate logit), E <= 1024, 1 <= K <= 8, 16 warps.
//   order: larger logit first, ties to the lower index (an order-preserving
//   integer key per logit, so the set and its order are the same as the
//   router kernel's per-warp selection).
//   T = the K-th largest of the 16 per-warp maxima: at least K logits are
//   >= T, so the top K are among the logits >= T. Every warp finds T from the
//   maxima and appends its logits >= T to a candidate list (typically a few);
//   warp 0 then takes K rounds of max, lowest index among equal keys, remove.
// Writes s_idx[0..K), s_l[0..K) = the selected logits and s_l[K] = lg[E]
// (read by block_topk_weights, so lg may be overwritten after the call).
// `scratch` holds topk_scratch_ints(E) ints. Ends with __syncthreads().
static __device__ void block_topk_select(const float* lg, int* scratch, int E, int K, bool has_gate, int* s_idx,
                                         float* s_l) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* wmax = scratch;        // [16] per-warp maxima
  int* ncand = scratch + 16;  // candidate count
  int* ck = scratch + 32;     // [E] candidate keys
  int* ci = ck + E;           // [E] candidate indices
  const int e0 = warp * 64 + lane, e1 = e0 + 32;
  const int k0 = e0 < E ? fkey(lg[e0]) : INT_MIN;
  const int k1 = e1 < E ? fkey(lg[e1]) : INT_MIN;
  const int m = redux_max(max(k0, k1));
  if (lane == 0) wmax[warp] = m;
  if (tid == 0) *ncand = 0;
  __syncthreads();
  // T: the maximum whose rank (larger first, then lower warp) is K - 1
  const int mine = lane < kTopkWarps ? wmax[lane] : INT_MIN;
  int rank = 0;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    const int v = wmax[w];
    rank += (v > mine) || (v == mine && w < lane);
  }
  const unsigned bt = __ballot_sync(kFull, lane < kTopkWarps && rank == K - 1);
  const int T = __shfl_sync(kFull, mine, __ffs(bt) - 1);
  const bool c0 = e0 < E && k0 >= T, c1 = e1 < E && k1 >= T;
  const unsigned b0 = __ballot_sync(kFull, c0), b1 = __ballot_sync(kFull, c1);
  int base = 0;
  if (lane == 0 && (b0 | b1)) base = atomicAdd(ncand, __popc(b0) + __popc(b1));
  base = __shfl_sync(kFull, base, 0);
  const unsigned below = (1u << lane) - 1u;
  if (c0) {
    const int q = base + __popc(b0 & below);
    ck[q] = k0;
    ci[q] = e0;
  }
  if (c1) {
    const int q = base + __popc(b0) + __popc(b1 & below);
    ck[q] = k1;
    ci[q] = e1;
  }
  __syncthreads();
  if (warp == 0) {
    const int n = *ncand;  // >= K
    int sel = 0;
    if (n <= 32) {
      int kk = lane < n ? ck[lane] : INT_MIN;
      const int ii = lane < n ? ci[lane] : INT_MAX;
      for (int k = 0; k < K; ++k) {
        const int best = redux_max(kk);
        const int bi = redux_min(kk == best ? ii : INT_MAX);
        if (ii == bi) kk = INT_MIN;
        if (lane == k) sel = bi;
      }
    } else {
      sel = topk_many_candidates(ck, ci, n, K, lane);
    }
    if (lane < K) {
      s_idx[lane] = sel;
      s_l[lane] = lg[sel];
    }
    if (lane == K) s_l[K] = has_gate ? lg[E] : 0.f;
  }
  __syncthreads();
}

// One warp: the routing weights of the selection (s_l from block_topk_select).
//   Softmax over all E logits followed by renormalisation over the selected K
//   equals a softmax over the selected logits alone (the full denominator
//   cancels): w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0), l_0 the largest,
//   the sum taken in k order exactly as the router kernel does (lane k
//   computes exp for slot k). s_w[K] = sigmoid(shared-gate logit), or 1.
static __device__ void block_topk_weights(const float* s_l, int K, bool has_gate, float* s_w) {
  const int lane = threadIdx.x & 31;
  const float pk = lane < K ? expf(s_l[lane < K ? lane : 0] - s_l[0]) : 0.f;
  float ps = 0.f;
  for (int k = 0; k < K; ++k) ps += __shfl_sync(kFull, pk, k);
  if (lane < K) s_w[lane] = pk / ps;
  if (lane == K) s_w[K] = has_gate ? 1.f / (1.f + expf(-s_l[K])) : 1.f;
}

// Selection and weights together (s_l: K + 1 floats of shared memory).
static __device__ void block_topk(const float* lg, int* scratch, int E, int K, bool has_gate, int* s_idx, float* s_l,
                                  float* s_w) {
  block_topk_select(lg, scratch, E, K, has_gate, s_idx, s_l);
  if ((threadIdx.x >> 5) == 0) block_topk_weights(s_l, K, has_gate, s_w);
  __syncthreads();
}

}  // namespace bgq
