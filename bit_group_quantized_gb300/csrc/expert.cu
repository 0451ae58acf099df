// expert.cu — grouped SwiGLU experts, combine, RMSNorm and residual add.
//
// Flash-MoE page, section "架构设计：SSD当显存用": CMD3 is the selected experts'
// forward pass, the combine and the norm. An expert is SwiGLU:
//   h = silu(gate x) * (up x)   (kept in fp32),   y = down h.
// The kernels run a plan of grouped-GEMV tasks (route.cu): one task is one
// expert applied to up to 8 tokens, so each weight row is read once for all of
// them. Rows are split across CTAs; the CTA stages its task's inputs once and
// keeps them while consecutive work items stay on the same task.
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kExpThreads = 256;
constexpr int kExpWarps = 8;
constexpr int kMaxNitE = 4;  // parts per lane and row-dot held in registers

__device__ __forceinline__ ExpertRef resolve(const ExpertSet& es, int e) {
  if (e < 0) return es.shared;
  ExpertRef r;
  const long long mw = (long long)es.d * es.f * es.bits / 32;  // words per matrix
  const long long mg = (long long)es.d * es.f / kGroup * 2;    // bf16 per matrix
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

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

template <int BITS>
__device__ __forceinline__ void load_row(const uint32_t* qrow, const uint32_t* sbrow, const RowGeo& rg, int lp,
                                         int it0, bool valid, uint4 (&qv)[kMaxNitE], uint32_t (&sv)[kMaxNitE]) {
#pragma unroll
  for (int i = 0; i < kMaxNitE; ++i) {
    int it = it0 + i;
    if (valid && it < rg.NIT) {
      int p = it * rg.LPR + lp;
      qv[i] = ldg_stream16(qrow + 4 * p);
      sv[i] = ldg_stream4(sbrow + part_group<BITS>(p));
    } else {
      qv[i] = make_uint4(0, 0, 0, 0);
      sv[i] = 0;
    }
  }
}

// Accumulate the parts of one load round into acc[t] for t < ntok.
template <int BITS>
__device__ __forceinline__ void dot_round(const uint4 (&qv)[kMaxNitE], const uint32_t (&sv)[kMaxNitE],
                                          const XStage& st, const RowGeo& rg, int lp, int it0, int ntok,
                                          float (&acc)[kTaskTok]) {
#pragma unroll
  for (int i = 0; i < kMaxNitE; ++i) {
    int it = it0 + i;
    if (it < rg.NIT) {
#pragma unroll
      for (int t = 0; t < kTaskTok; ++t)
        if (t < ntok) acc[t] = part_dot24<BITS>(qv[i], sv[i], st, t, it, lp, rg, acc[t]);
    }
  }
}

struct ItemRange {
  int begin, end;
};
__device__ __forceinline__ ItemRange my_items(int total) {
  int per = (total + gridDim.x - 1) / gridDim.x;
  int b = blockIdx.x * per;
  int e = b + per;
  return ItemRange{b < total ? b : total, e < total ? e : total};
}

// ---------------------------------------------------------------------------
// gate/up + SiLU*mul. Item = (task, block of rows of d_ff).
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kExpThreads)
k_gateup(ExpertSet es, const Plan* __restrict__ plan, const uint16_t* __restrict__ x, float* __restrict__ H,
         int nslot) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_off[kTaskTok];
  const int d = es.d, f = es.f;
  const RowGeo rg = row_geo(d, BITS);
  const int rows_item = kExpWarps * rg.RPP;
  const int nrb = (f + rows_item - 1) / rows_item;
  const int total = plan->ntasks * nrb;
  const ItemRange ir = my_items(total);
  const XStage st = xstage_carve(smem, kTaskTok, d);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rs = lane / rg.LPR, lp = lane - rs * rg.LPR;
  const int wpr = d * BITS / 32, gpr = d / kGroup;
  int staged = -1;
  for (int item = ir.begin; item < ir.end; ++item) {
    const int ti = item / nrb, rb = item - ti * nrb;
    const Task& tk = plan_tasks(plan)[ti];
    const int ntok = tk.ntok;
    const ExpertRef ex = resolve(es, tk.expert);
    const int row = rb * rows_item + warp * rg.RPP + rs;
    const bool valid = row < f;
    const uint32_t* gq = ex.gate_q + (size_t)(valid ? row : 0) * wpr;
    const uint32_t* uq = ex.up_q + (size_t)(valid ? row : 0) * wpr;
    const uint32_t* gs = reinterpret_cast<const uint32_t*>(ex.gate_sb) + (size_t)(valid ? row : 0) * gpr;
    const uint32_t* us = reinterpret_cast<const uint32_t*>(ex.up_sb) + (size_t)(valid ? row : 0) * gpr;
    uint4 gqv[kMaxNitE], uqv[kMaxNitE];
    uint32_t gsv[kMaxNitE], usv[kMaxNitE];
    load_row<BITS>(gq, gs, rg, lp, 0, valid, gqv, gsv);
    load_row<BITS>(uq, us, rg, lp, 0, valid, uqv, usv);
    if (ti != staged) {
      __syncthreads();  // previous item finished reading the staged inputs
      if (threadIdx.x < kTaskTok) s_off[threadIdx.x] = threadIdx.x < ntok ? tk.tok[threadIdx.x] * d : 0;
      __syncthreads();
      stage_x24<BITS>(GatherSrc<uint16_t>{x, s_off}, ntok, d, st);
      staged = ti;
    }
    float ga[kTaskTok], ua[kTaskTok];
#pragma unroll
    for (int t = 0; t < kTaskTok; ++t) ga[t] = ua[t] = 0.f;
    for (int it0 = 0; it0 < rg.NIT; it0 += kMaxNitE) {
      if (it0 > 0) {
        load_row<BITS>(gq, gs, rg, lp, it0, valid, gqv, gsv);
        load_row<BITS>(uq, us, rg, lp, it0, valid, uqv, usv);
      }
      dot_round<BITS>(gqv, gsv, st, rg, lp, it0, ntok, ga);
      dot_round<BITS>(uqv, usv, st, rg, lp, it0, ntok, ua);
    }
#pragma unroll
    for (int t = 0; t < kTaskTok; ++t) {
      if (t < ntok) {
        float g = row_reduce(ga[t], rg.LPR), u = row_reduce(ua[t], rg.LPR);
        if (valid && lp == 0) H[((size_t)tk.tok[t] * nslot + tk.slot[t]) * f + row] = silu_f(g) * u;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// down projection. Item = (task, block of rows of d_model).
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kExpThreads)
k_down(ExpertSet es, const Plan* __restrict__ plan, const float* __restrict__ H, float* __restrict__ Y, int nslot) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_off[kTaskTok];
  const int d = es.d, f = es.f;
  const RowGeo rg = row_geo(f, BITS);
  const int rows_item = kExpWarps * rg.RPP;
  const int nrb = (d + rows_item - 1) / rows_item;
  const int total = plan->ntasks * nrb;
  const ItemRange ir = my_items(total);
  const XStage st = xstage_carve(smem, kTaskTok, f);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rs = lane / rg.LPR, lp = lane - rs * rg.LPR;
  const int wpr = f * BITS / 32, gpr = f / kGroup;
  int staged = -1;
  for (int item = ir.begin; item < ir.end; ++item) {
    const int ti = item / nrb, rb = item - ti * nrb;
    const Task& tk = plan_tasks(plan)[ti];
    const int ntok = tk.ntok;
    const ExpertRef ex = resolve(es, tk.expert);
    const int row = rb * rows_item + warp * rg.RPP + rs;
    const bool valid = row < d;
    const uint32_t* dq = ex.down_q + (size_t)(valid ? row : 0) * wpr;
    const uint32_t* ds = reinterpret_cast<const uint32_t*>(ex.down_sb) + (size_t)(valid ? row : 0) * gpr;
    uint4 qv[kMaxNitE];
    uint32_t sv[kMaxNitE];
    load_row<BITS>(dq, ds, rg, lp, 0, valid, qv, sv);
    if (ti != staged) {
      __syncthreads();
      if (threadIdx.x < kTaskTok)
        s_off[threadIdx.x] = threadIdx.x < ntok ? (tk.tok[threadIdx.x] * nslot + tk.slot[threadIdx.x]) * f : 0;
      __syncthreads();
      stage_x24<BITS>(GatherSrc<float>{H, s_off}, ntok, f, st);
      staged = ti;
    }
    float acc[kTaskTok];
#pragma unroll
    for (int t = 0; t < kTaskTok; ++t) acc[t] = 0.f;
    for (int it0 = 0; it0 < rg.NIT; it0 += kMaxNitE) {
      if (it0 > 0) load_row<BITS>(dq, ds, rg, lp, it0, valid, qv, sv);
      dot_round<BITS>(qv, sv, st, rg, lp, it0, ntok, acc);
    }
#pragma unroll
    for (int t = 0; t < kTaskTok; ++t) {
      if (t < ntok) {
        float v = row_reduce(acc[t], rg.LPR);
        if (valid && lp == 0) Y[((size_t)tk.tok[t] * nslot + tk.slot[t]) * d + row] = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Small batches (all inputs fit in shared memory): one 512-thread CTA per SM
// stages every token's input once, then walks its share of the rows of every
// task. A warp keeps the weight rows of its next work item in flight while it
// computes the current one, so each SM has ~100 KB of row loads outstanding
// (the HBM latency-bandwidth product per SM), and no CTA restages inputs when
// the task changes. Per-row arithmetic (part order, accumulation, butterfly)
// is the same as in k_gateup / k_down and the persistent kernel, so results
// are bit-identical across the three.
// ---------------------------------------------------------------------------
constexpr int kAllThreads = 384;  // 12 warps: two work items of row loads per warp fit in registers
constexpr int kAllWarps = kAllThreads / 32;
constexpr int kAllRows = 8;  // rows per down-projection work item

struct RowSpan {
  int b, e;
};
__device__ __forceinline__ RowSpan cta_rows(int n) {
  return RowSpan{(int)((long long)n * blockIdx.x / gridDim.x), (int)((long long)n * (blockIdx.x + 1) / gridDim.x)};
}

// Gate and up rows (all parts of one row per lane group; d-rows have LPR = 32).
struct GateUpRows {
  uint4 g[kMaxNitE], u[kMaxNitE];
  uint32_t gs[kMaxNitE], us[kMaxNitE];
};

// The plan's tasks, or without a plan (one explicit expert over B tokens):
// tasks of 8 consecutive tokens of the shared-expert view in slot 0, the
// tasks k_plan_single would build, written to s_task (ends with a block
// barrier then).
__device__ __forceinline__ const Task* tasks_of(const Plan* plan, int B, Task* s_task, int& ntasks) {
  if (plan) {
    ntasks = plan->ntasks;
    return plan_tasks(plan);
  }
  ntasks = (B + kTaskTok - 1) / kTaskTok;
  for (int c = threadIdx.x; c < ntasks; c += blockDim.x) {
    Task& tk = s_task[c];
    tk.expert = -1;
    tk.ntok = min(kTaskTok, B - c * kTaskTok);
    for (int i = 0; i < kTaskTok; ++i) {
      tk.tok[i] = c * kTaskTok + i;
      tk.slot[i] = 0;
    }
  }
  __syncthreads();
  return s_task;
}

template <int BITS>
__device__ __forceinline__ void load_gateup(const ExpertSet& es, const Task* tasks, int item, int nr, int r0,
                                            const RowGeo& rg, int lane, GateUpRows& R) {
  const Task& tk = tasks[item / nr];
  const int row = r0 + item % nr;
  const ExpertRef ex = resolve(es, tk.expert);
  const int wpr = es.d * BITS / 32, gpr = es.d / kGroup;
  load_row<BITS>(ex.gate_q + (size_t)row * wpr, reinterpret_cast<const uint32_t*>(ex.gate_sb) + (size_t)row * gpr,
                 rg, lane, 0, true, R.g, R.gs);
  load_row<BITS>(ex.up_q + (size_t)row * wpr, reinterpret_cast<const uint32_t*>(ex.up_sb) + (size_t)row * gpr, rg,
                 lane, 0, true, R.u, R.us);
}

template <int BITS>
__global__ void __launch_bounds__(kAllThreads, 1)
k_gateup_all(ExpertSet es, const Plan* __restrict__ plan, const uint16_t* __restrict__ x, int B,
             float* __restrict__ H, int nslot, XStage gst) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Task s_task[kPlanlessTasks];
  pdl_wait();     // launched as a programmatic dependent: nothing is touched before the earlier kernels end
  pdl_trigger();
  int ntasks;
  const Task* tasks = tasks_of(plan, B, s_task, ntasks);
  const int d = es.d, f = es.f;
  const RowGeo rg = row_geo(d, BITS);  // LPR == 32, NIT <= kMaxNitE (checked by the launcher)
  // inputs staged here, or (too many tokens for shared memory) read from the
  // copy k_stage_tokens made in global memory (L1/L2 resident)
  const bool local = gst.chunks == nullptr;
  XStage st = gst;
  if (local) {
    st = xstage_carve(smem, B, d);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RowSpan rs = cta_rows(f);
  const int nr = rs.e - rs.b;
  const int total = ntasks * nr;
  GateUpRows cur, nxt;
  if (warp < total) load_gateup<BITS>(es, tasks, warp, nr, rs.b, rg, lane, cur);  // in flight during staging
  if (local) stage_x24_pairs<BITS>(StridedSrc<uint16_t>{x, d}, B, d, st);  // two code words per thread
  for (int item = warp; item < total; item += kAllWarps) {
    if (item + kAllWarps < total) load_gateup<BITS>(es, tasks, item + kAllWarps, nr, rs.b, rg, lane, nxt);
    const Task& tk = tasks[item / nr];
    const int row = rs.b + item % nr;
    for (int i = 0; i < tk.ntok; ++i) {
      const int t = tk.tok[i];
      float ga = 0.f, ua = 0.f;
#pragma unroll
      for (int it = 0; it < kMaxNitE; ++it) {
        if (it < rg.NIT) {
          uint4 xc[4 * Geo<BITS>::kNch];
          uint2 xh[4 * Geo<BITS>::kNch];
          load_part_x<BITS>(st, t, it, lane, rg, xc, xh);
          const float2 pi = st.partinfo[t * rg.P + it * 32 + lane];
          ga = part_dot_x<BITS>(cur.g[it], cur.gs[it], xc, xh, pi, ga);
          ua = part_dot_x<BITS>(cur.u[it], cur.us[it], xc, xh, pi, ua);
        }
      }
      ga = warp_sum(ga);
      ua = warp_sum(ua);
      if (lane == 0) H[((size_t)t * nslot + tk.slot[i]) * f + row] = silu_f(ga) * ua;
    }
    cur = nxt;
  }
}

// Up to kAllRows down rows of one task (f-rows: one part per lane, RPP rows per warp pass).
struct DownRows {
  uint4 q[kAllRows];
  uint32_t s[kAllRows];
};

// Work item i: task i / nch, row groups [g0, g1) of the CTA's rows (chunks of
// at most kAllRows row groups, near-equal sizes).
struct DownItem {
  int task, g0, g1;
};
__device__ __forceinline__ DownItem down_item(int i, int nch, int nrg) {
  const int ti = i / nch, ci = i - ti * nch;
  return DownItem{ti, nrg * ci / nch, nrg * (ci + 1) / nch};
}

template <int BITS>
__device__ __forceinline__ void load_down(const ExpertSet& es, const Task* tasks, const DownItem& it, int r0, int nrows,
                                          const RowGeo& rg, int lp, int rsub, DownRows& R) {
  const ExpertRef ex = resolve(es, tasks[it.task].expert);
  const int wpr = es.f * BITS / 32, gpr = es.f / kGroup;
#pragma unroll
  for (int u = 0; u < kAllRows; ++u) {
    const int r = (it.g0 + u) * rg.RPP + rsub;  // local row
    if (it.g0 + u < it.g1 && r < nrows) {
      const size_t row = (size_t)(r0 + r);
      R.q[u] = ldg_stream16(ex.down_q + row * wpr + 4 * lp);
      R.s[u] = ldg_stream4(reinterpret_cast<const uint32_t*>(ex.down_sb) + row * gpr + part_group<BITS>(lp));
    } else {
      R.q[u] = make_uint4(0, 0, 0, 0);
      R.s[u] = 0;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kAllThreads, 1)
k_down_all(ExpertSet es, const Plan* __restrict__ plan, const float* __restrict__ H, int B,
           float* __restrict__ Y, int nslot, XStage gst, Combine cb) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Task s_task[kPlanlessTasks];
  pdl_wait();  // as k_gateup_all
  pdl_trigger();
  int ntasks;
  const Task* tasks = tasks_of(plan, B, s_task, ntasks);
  const int d = es.d, f = es.f;
  const RowGeo rg = row_geo(f, BITS);  // NIT == 1 (checked by the launcher)
  const int T = B * nslot;             // staged vector (tok, slot) at index tok * nslot + slot
  const bool local = gst.chunks == nullptr;  // else: staged in global memory (see k_gateup_all)
  XStage st = gst;
  if (local) {
    st = xstage_carve(smem, T, f);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lp = lane % rg.LPR, rsub = lane / rg.LPR;
  const RowSpan rs = cta_rows(d);
  const int nrows = rs.e - rs.b;
  const int nrg = (nrows + rg.RPP - 1) / rg.RPP;
  const int nch = (nrg + kAllRows - 1) / kAllRows;
  const int total = ntasks * nch;
  DownRows cur, nxt;
  if (warp < total) load_down<BITS>(es, tasks, down_item(warp, nch, nrg), rs.b, nrows, rg, lp, rsub, cur);
  if (local) stage_x24_pairs<BITS>(StridedSrc<float>{H, f}, T, f, st);
  for (int i = warp; i < total; i += kAllWarps) {
    if (i + kAllWarps < total)
      load_down<BITS>(es, tasks, down_item(i + kAllWarps, nch, nrg), rs.b, nrows, rg, lp, rsub, nxt);
    const DownItem it = down_item(i, nch, nrg);
    const Task& tk = tasks[it.task];
    for (int j = 0; j < tk.ntok; ++j) {
      const int v = tk.tok[j] * nslot + tk.slot[j];
      uint4 xc[4 * Geo<BITS>::kNch];
      uint2 xh[4 * Geo<BITS>::kNch];
      load_part_x<BITS>(st, v, 0, lp, rg, xc, xh);
      const float2 pi = st.partinfo[v * rg.P + lp];
      float acc[kAllRows];
#pragma unroll
      for (int u = 0; u < kAllRows; ++u) acc[u] = part_dot_x<BITS>(cur.q[u], cur.s[u], xc, xh, pi, 0.f);
      float* yv = Y + (size_t)v * d + rs.b;
      if (rg.LPR >= 8) {
        const float y = row_reduce8(acc, rg.LPR, lane);
        const int o1 = rg.LPR >> 1, o2 = o1 >> 1, o3 = o2 >> 1;
        if ((lp & (o3 - 1)) == 0) {
          const int u = ((lp & o1) ? 4 : 0) + ((lp & o2) ? 2 : 0) + ((lp & o3) ? 1 : 0);
          const int r = (it.g0 + u) * rg.RPP + rsub;
          if (it.g0 + u < it.g1 && r < nrows) yv[r] = y;
        }
      } else {
#pragma unroll
        for (int u = 0; u < kAllRows; ++u) {
          const float y = row_reduce(acc[u], rg.LPR);
          const int r = (it.g0 + u) * rg.RPP + rsub;
          if (lp == 0 && it.g0 + u < it.g1 && r < nrows) yv[r] = y;
        }
      }
    }
    cur = nxt;
  }
  if (cb.out || cb.out_f32) {
    // This CTA now holds every (token, slot) output of its rows (the
    // tensor-core tasks' ran before this kernel): the weighted combine of
    // k_combine, same order (k = 0..K-1, then the shared expert).
    __syncthreads();
    for (int i = threadIdx.x; i < B * nrows; i += blockDim.x) {
      const int t = i / nrows, r = rs.b + (i - t * nrows);
      const float* yt = Y + (size_t)t * nslot * d + r;
      float acc = 0.f;
      for (int k = 0; k < cb.K; ++k) acc = fmaf(cb.w[t * cb.K + k], yt[(size_t)k * d], acc);
      const float g = cb.gamma ? cb.gamma[t] : 1.f;
      acc = fmaf(g, yt[(size_t)cb.K * d], acc);
      if (cb.out) cb.out[(size_t)t * d + r] = f2bf(acc);
      if (cb.out_f32) cb.out_f32[(size_t)t * d + r] = acc;
    }
  }
}

// T staged vectors of `cols` values: bytes (shared or global memory).
static size_t all_smem(int cols, int bits, int T) { return xstage_bytes(T, cols, bits); }
constexpr size_t kAllSmemMax = 200 * 1024;

size_t staged_tokens_bytes(int cols, int bits, int T) { return all_smem(cols, bits, T); }

// Stages T vectors of `cols` values into global memory (same layout and
// values as the shared-memory staging), one thread per code word.
template <int BITS, typename Src>
__global__ void k_stage_tokens(const Src src, int T, int cols, XStage st) {
  using G = Geo<BITS>;
  const RowGeo rg = row_geo(cols, BITS);
  const int words = cols * BITS / 32;
  const int tw = blockIdx.x * blockDim.x + threadIdx.x;  // whole warps run: groups never straddle one
  const bool active = tw < T * words;
  const int t = active ? tw / words : 0, w = active ? tw - t * words : 0;
  float v[G::kPer];
#pragma unroll
  for (int i = 0; i < G::kPer; i += 8) {
    if (active) {
      src.load8(t, w * G::kPer + i, v + i);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[i + j] = 0.f;
    }
  }
  stage_word<BITS>(v, active, t, w, rg, __ffs(rg.LPR) - 1, st);
}

static XStage global_stage(unsigned char* buf, int cols, int T) { return xstage_carve(buf, T, cols); }
template <int BITS, typename Src>
static cudaError_t stage_tokens(const Src src, int T, int cols, XStage st, cudaStream_t s) {
  const int n = T * (cols * BITS / 32);
  k_stage_tokens<BITS><<<(n + 255) / 256, 256, 0, s>>>(src, T, cols, st);
  return cudaGetLastError();
}

template <typename K>
static cudaError_t set_smem(K kern, size_t sm) {
  if (sm > 48 * 1024) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  return cudaSuccess;
}

static int expert_grid(int max_items) {
  int g = num_sms() * 2;
  return max_items < g ? (max_items > 0 ? max_items : 1) : g;
}

bool grouped_planless_ok(const ExpertSet& es, int batch, bool stage_ws) {
  const RowGeo rg = row_geo(es.d, es.bits), rf = row_geo(es.f, es.bits);
  if (batch > kPlanlessTasks * kTaskTok) return false;
  const bool gu = rg.LPR == 32 && rg.NIT <= kMaxNitE && (all_smem(es.d, es.bits, batch) <= kAllSmemMax || stage_ws);
  const bool dn = rf.NIT == 1 && (all_smem(es.f, es.bits, batch) <= kAllSmemMax || stage_ws);
  return gu && dn;
}

cudaError_t launch_gateup(const ExpertSet& es, const Plan* plan, int max_tasks, int batch, const uint16_t* x, float* H,
                          int nslot, unsigned char* stage_ws, cudaStream_t s) {
  RowGeo rg = row_geo(es.d, es.bits);
  const bool fits = all_smem(es.d, es.bits, batch) <= kAllSmemMax;
  if (!plan && !grouped_planless_ok(es, batch, stage_ws != nullptr)) return cudaErrorInvalidValue;
  if (rg.LPR == 32 && rg.NIT <= kMaxNitE && (fits || stage_ws)) {
    XStage gst{};
    size_t sm = 0;
    cudaError_t e;
    if (fits) {
      sm = all_smem(es.d, es.bits, batch);
    } else {
      gst = global_stage(stage_ws, es.d, batch);
      e = es.bits == 4 ? stage_tokens<4>(StridedSrc<uint16_t>{x, es.d}, batch, es.d, gst, s)
                       : stage_tokens<2>(StridedSrc<uint16_t>{x, es.d}, batch, es.d, gst, s);
      if (e != cudaSuccess) return e;
    }
    if (es.bits == 4) {
      if ((e = set_smem(k_gateup_all<4>, sm)) != cudaSuccess) return e;
      e = launch_overlapped(k_gateup_all<4>, num_sms(), kAllThreads, sm, s, es, plan, x, batch, H, nslot, gst);
      if (e != cudaSuccess) return e;
    } else {
      if ((e = set_smem(k_gateup_all<2>, sm)) != cudaSuccess) return e;
      e = launch_overlapped(k_gateup_all<2>, num_sms(), kAllThreads, sm, s, es, plan, x, batch, H, nslot, gst);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  size_t sm = qgemv_int_smem(es.d, es.bits, kTaskTok);
  int nrb = (es.f + kExpWarps * rg.RPP - 1) / (kExpWarps * rg.RPP);
  int grid = expert_grid(max_tasks * nrb);
  cudaError_t e;
  if (es.bits == 4) {
    if ((e = set_smem(k_gateup<4>, sm)) != cudaSuccess) return e;
    k_gateup<4><<<grid, kExpThreads, sm, s>>>(es, plan, x, H, nslot);
  } else {
    if ((e = set_smem(k_gateup<2>, sm)) != cudaSuccess) return e;
    k_gateup<2><<<grid, kExpThreads, sm, s>>>(es, plan, x, H, nslot);
  }
  return cudaGetLastError();
}

cudaError_t launch_down(const ExpertSet& es, const Plan* plan, int max_tasks, int batch, const float* H, float* Y,
                        int nslot, unsigned char* stage_ws, const Combine& cb, cudaStream_t s) {
  RowGeo rg = row_geo(es.f, es.bits);
  const int T = batch * nslot;
  const bool fits = all_smem(es.f, es.bits, T) <= kAllSmemMax;
  if (!plan && (nslot != 1 || !grouped_planless_ok(es, batch, stage_ws != nullptr))) return cudaErrorInvalidValue;
  if (rg.NIT == 1 && (fits || stage_ws)) {
    XStage gst{};
    size_t sm = 0;
    cudaError_t e;
    if (fits) {
      sm = all_smem(es.f, es.bits, T);
    } else {
      gst = global_stage(stage_ws, es.f, T);
      e = es.bits == 4 ? stage_tokens<4>(StridedSrc<float>{H, es.f}, T, es.f, gst, s)
                       : stage_tokens<2>(StridedSrc<float>{H, es.f}, T, es.f, gst, s);
      if (e != cudaSuccess) return e;
    }
    if (es.bits == 4) {
      if ((e = set_smem(k_down_all<4>, sm)) != cudaSuccess) return e;
      e = launch_overlapped(k_down_all<4>, num_sms(), kAllThreads, sm, s, es, plan, H, batch, Y, nslot, gst, cb);
      if (e != cudaSuccess) return e;
    } else {
      if ((e = set_smem(k_down_all<2>, sm)) != cudaSuccess) return e;
      e = launch_overlapped(k_down_all<2>, num_sms(), kAllThreads, sm, s, es, plan, H, batch, Y, nslot, gst, cb);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  size_t sm = qgemv_int_smem(es.f, es.bits, kTaskTok);
  int nrb = (es.d + kExpWarps * rg.RPP - 1) / (kExpWarps * rg.RPP);
  int grid = expert_grid(max_tasks * nrb);
  cudaError_t e;
  if (es.bits == 4) {
    if ((e = set_smem(k_down<4>, sm)) != cudaSuccess) return e;
    k_down<4><<<grid, kExpThreads, sm, s>>>(es, plan, H, Y, nslot);
  } else {
    if ((e = set_smem(k_down<2>, sm)) != cudaSuccess) return e;
    k_down<2><<<grid, kExpThreads, sm, s>>>(es, plan, H, Y, nslot);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (cb.out || cb.out_f32)  // the per-task kernel leaves the combine to its own launch
    return launch_combine(Y, cb.w, cb.gamma, batch, cb.K, es.d, cb.out, cb.out_f32, s);
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// combine, RMSNorm, residual
// ---------------------------------------------------------------------------
__global__ void k_combine(const float* __restrict__ Y, const float* __restrict__ w, const float* __restrict__ gamma,
                          int B, int K, int d, uint16_t* __restrict__ out, float* __restrict__ out_f32) {
  const long long n = (long long)B * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / d), r = (int)(i - (long long)t * d);
    const float* yt = Y + (size_t)t * (K + 1) * d + r;
    float acc = 0.f;
    for (int k = 0; k < K; ++k) acc = fmaf(w[t * K + k], yt[(size_t)k * d], acc);
    const float g = gamma ? gamma[t] : 1.f;
    acc = fmaf(g, yt[(size_t)K * d], acc);
    if (out) out[i] = f2bf(acc);
    if (out_f32) out_f32[i] = acc;
  }
}

cudaError_t launch_combine(const float* Y, const float* w, const float* gamma, int batch, int K, int d,
                           uint16_t* out, float* out_f32, cudaStream_t s) {
  long long n = (long long)batch * d;
  int grid = (int)((n + 255) / 256);
  int cap = num_sms() * 8;
  if (grid > cap) grid = cap;
  k_combine<<<grid, 256, 0, s>>>(Y, w, gamma, batch, K, d, out, out_f32);
  return cudaGetLastError();
}

// One CTA per token: a = bf16(h * (1/sqrt(mean(h^2) + eps)) * rho); h fp32,
// or bf16 widened exactly (the same bits as on the widened copy). Launched as
// a programmatic dependent: it waits before touching memory.
__device__ __forceinline__ float rms_ld(const float* p) { return *p; }
__device__ __forceinline__ float rms_ld(const uint16_t* p) { return bf16f(*p); }
template <typename T>
__global__ void __launch_bounds__(256) k_rmsnorm(const T* __restrict__ h, const uint16_t* __restrict__ rho, int d,
                                                 float eps, uint16_t* __restrict__ a) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  const T* ht = h + (size_t)blockIdx.x * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = rms_ld(ht + i);
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  const float r = 1.f / sqrtf(tot / (float)d + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float v = rms_ld(ht + i) * r;
    if (rho) v *= bf16f(rho[i]);
    a[(size_t)blockIdx.x * d + i] = f2bf(v);
  }
}

cudaError_t launch_rmsnorm(const float* h, const uint16_t* rho, int batch, int d, float eps, uint16_t* a,
                           cudaStream_t s) {
  return launch_overlapped(k_rmsnorm<float>, batch, 256, 0, s, h, rho, d, eps, a);
}
cudaError_t launch_rmsnorm_bf16(const uint16_t* x, const uint16_t* rho, int batch, int d, float eps, uint16_t* a,
                                cudaStream_t s) {
  return launch_overlapped(k_rmsnorm<uint16_t>, batch, 256, 0, s, x, rho, d, eps, a);
}

__global__ void k_residual(float* __restrict__ h, const float* __restrict__ delta, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    h[i] += delta[i];
}

cudaError_t launch_residual_add(float* h, const float* delta, long long n, cudaStream_t s) {
  int grid = (int)((n + 255) / 256);
  int cap = num_sms() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  k_residual<<<grid, 256, 0, s>>>(h, delta, n);
  return cudaGetLastError();
}

__global__ void k_widen(const uint16_t* __restrict__ x, float* __restrict__ h, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) h[i] = bf16f(x[i]);
}

cudaError_t launch_widen(const uint16_t* x, float* h, int n, cudaStream_t s) {
  int grid = (n + 255) / 256;
  if (grid > 1024) grid = 1024;
  k_widen<<<grid, 256, 0, s>>>(x, h, n);
  return cudaGetLastError();
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 132;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 132;
  return n;
}

}  // namespace bgq
