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

// Top-K selection, run by every CTA on the logits in shared memory (lg[0..E),
// lg[E] = shared-gate logit), E <= 1024, K <= 8.
//   selection: order (larger logit, then lower index) — a total order, so the
//   set and its order are the same as the router kernel's per-warp selection.
//   Each warp takes the top K of its 64 logits (K rounds of redux.sync on an
//   order-preserving integer key, ties to the lowest index), then warp 0
//   merges the 16 x K candidates the same way.
//   weights: softmax over all E logits followed by renormalisation over the
//   selected K equals a softmax over the selected logits alone (the full
//   denominator cancels), so w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0) with
//   l_0 the largest logit, summed in k order exactly as the router kernel does.
// Writes s_idx[0..K), s_w[0..K) and s_w[K] = gamma. `cand` holds 2*16*8 ints.
static __device__ void block_topk(const float* lg, int* cand, int E, int K, bool has_gate, int* s_idx, float* s_w) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* cand_k = cand;                  // [16][8] keys
  int* cand_i = cand_k + kTopkWarps * 8;  // [16][8] indices
  // this warp's elements: e0 = warp*64 + lane, e1 = e0 + 32
  const int e0 = warp * 64 + lane, e1 = e0 + 32;
  int k0 = e0 < E ? fkey(lg[e0]) : INT_MIN;
  int k1 = e1 < E ? fkey(lg[e1]) : INT_MIN;
  for (int k = 0; k < K; ++k) {
    const int best = redux_max(max(k0, k1));
    const int i0 = (k0 == best && e0 < E) ? e0 : INT_MAX;
    const int i1 = (k1 == best && e1 < E) ? e1 : INT_MAX;
    const int bi = redux_min(min(i0, i1));
    if (lane == 0) {
      cand_k[warp * 8 + k] = best;
      cand_i[warp * 8 + k] = bi;
    }
    if (bi == e0) k0 = INT_MIN;
    if (bi == e1) k1 = INT_MIN;
  }
  __syncthreads();
  // merge: lane j of warp 0 holds candidate slots j, j+32, j+64, j+96 (slot = w*8 + k)
  if (warp == 0) {
    int ck[4], ci[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = j * 32 + lane;
      const bool ok = c < kTopkWarps * 8 && (c & 7) < K;
      ck[j] = ok ? cand_k[c] : INT_MIN;
      ci[j] = ok ? cand_i[c] : INT_MAX;
    }
    int mine = 0;
    for (int k = 0; k < K; ++k) {
      int lb = INT_MIN;
#pragma unroll
      for (int j = 0; j < 4; ++j) lb = max(lb, ck[j]);
      const int best = redux_max(lb);
      int li = INT_MAX;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ck[j] == best) li = min(li, ci[j]);
      const int bi = redux_min(li);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ci[j] == bi) ck[j] = INT_MIN;
      if (lane == k) mine = bi;
    }
    if (lane < K) s_idx[lane] = mine;
    __syncwarp();
    if (lane == 0) {
      float p[8], ps = 0.f;
      const float l0 = lg[s_idx[0]];
      for (int k = 0; k < K; ++k) {
        p[k] = expf(lg[s_idx[k]] - l0);
        ps += p[k];
      }
      for (int k = 0; k < K; ++k) s_w[k] = p[k] / ps;
      s_w[K] = has_gate ? 1.f / (1.f + expf(-lg[E])) : 1.f;
    }
  }
  __syncthreads();
}

}  // namespace bgq
