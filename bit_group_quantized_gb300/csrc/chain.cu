// chain.cu — a chain of dependent group-quantized GEMVs in one persistent
// launch: the rest of a decoder layer around the MoE block.
//
// Flash-MoE page, section "架构设计：SSD当显存用": besides the expert
// forward, every layer runs the attention input projections (CMD1) and the
// output projection with its norm (CMD2) on the GPU; in the 4-bit model these
// are group-quantized matrices like the experts'. The attention mixing between
// them is outside this library, so the chain composes what is left:
//     v_0 = norm ? bf16(rmsnorm(x) [* rho]) : x
//     v_i = bf16(W_i v_{i-1})                      i = 1..n
//     out = W_n v_{n-1}  (+ x when residual)       fp32, and its bf16
// One CTA per SM, cooperative launch. Step i: every CTA stages v_{i-1} (the
// normalised x for i = 1, computed redundantly but identically in every CTA;
// else the previous step's output from global memory) and computes its share
// of W_i's rows, every warp requesting up to four of its rows at once (a
// 4096-row step is a single round of loads); a grid-wide counter then orders
// the steps. The rows of step i+1 are requested before that wait, so their
// latency overlaps it.
// Per row the arithmetic is q4_gemv's (k_qgemv_int) and the norm is
// bgq_rmsnorm's (k_rmsnorm), so the chain gives the bits of the separate calls.
#include "../../include/bgq.h"
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kChThreads = 256;
constexpr int kChWarps = kChThreads / 32;
constexpr int kChNit = 4;  // parts per lane and row held in registers at once
constexpr int kChU = 4;    // row units per warp requested at once (a 4096-row step is one round)

struct ChainParams {
  ChainStep st[kMaxChain];
  int n;
  const uint16_t* x;  // bf16 [T][d]
  int norm;            // rmsnorm the input first
  const uint16_t* rho; // its weights (nullable: none)
  float eps;
  int residual;
  uint16_t* out;      // bf16 [T][rows_n] (nullable)
  float* out_f32;     // fp32 [T][rows_n] (nullable)
  uint16_t* buf[2];   // bf16 [T][ldb]: outputs of the inner steps
  int ldb;
  Ctrl* ctrl;
  int* counter;       // grid-wide arrivals (zero at launch)
  long long timeout_ns;
};

__device__ __forceinline__ int ch_ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ch_time() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Input of the first step: the normalised tokens, rounded to bf16 as
// bgq_rmsnorm writes them (r[t] = 1 / sqrt(mean(x_t^2) + eps)).
struct NormSrc {
  const uint16_t* x;
  int d;
  const float* r;
  const uint16_t* rho;
  __device__ void load8(int t, int k0, float* v) const {
    float h[8];
    load8_from(x + (size_t)t * d + k0, h);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a = h[j] * r[t];
      if (rho) a *= bf16f(rho[k0 + j]);
      v[j] = bf16f(f2bf(a));
    }
  }
};

// Input of the later steps: the previous step's outputs, written by other
// CTAs, read through L2 only (never from a stale L1 line).
struct ChainL2Src {
  const uint16_t* x;
  int ld;
  __device__ void load8(int t, int k0, float* v) const {
    unpack_bf16x8(__ldcg(reinterpret_cast<const uint4*>(x + (size_t)t * ld + k0)), v);
  }
};

// One warp's rows of a step: unit u = rows [u*RPP, u*RPP + RPP), this lane's
// row u*RPP + rs; the first kChNit parts of the row.
template <int BITS>
__device__ __forceinline__ void ch_load(const ChainStep& W, const RowGeo& rg, int unit, int rs, int lp, int it0,
                                        uint4 (&qv)[kChNit], uint32_t (&sv)[kChNit]) {
  const int row = unit * rg.RPP + rs;
  const bool valid = row < W.rows;
  const int wpr = W.cols * BITS / 32, gpr = W.cols / kGroup;
  const uint32_t* qrow = W.q + (size_t)(valid ? row : 0) * wpr;
  const uint32_t* sbrow = W.sb + (size_t)(valid ? row : 0) * gpr;
#pragma unroll
  for (int i = 0; i < kChNit; ++i) {
    const int it = it0 + i;
    if (it < rg.NIT && valid) {
      const int p = it * rg.LPR + lp;
      qv[i] = ldg_stream16(qrow + 4 * p);
      sv[i] = ldg_stream4(sbrow + part_group<BITS>(p));
    } else {
      qv[i] = make_uint4(0, 0, 0, 0);
      sv[i] = 0;
    }
  }
}

// Grid-wide wait: every CTA has finished step k. After the block barrier,
// thread 0 adds 1 to the counter with a release reduction (ordered after the
// CTA's stores, nothing to wait for) and polls it with acquire loads until
// every CTA of the grid has arrived (k + 1 arrivals each). False (for the
// whole CTA) on timeout or when another CTA gave up.
__device__ bool ch_grid_wait(const ChainParams& P, int k, int* s_fail) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(P.counter) : "memory");
    const int target = (k + 1) * (int)gridDim.x;
    const unsigned long long t0 = ch_time();
    int ok = 1;
    for (long long it = 1; ch_ld_acquire(P.counter) < target; ++it) {
      if ((it & 15) == 0) {
        if (*(volatile int*)&P.ctrl->misc[0] != 0 || (long long)(ch_time() - t0) > P.timeout_ns || it > (1ll << 26)) {
          atomicExch(&P.ctrl->status, BGQ_ERR_TIMEOUT);
          atomicExch(&P.ctrl->misc[0], 1);
          ok = 0;
          break;
        }
      }
    }
    *s_fail = !ok;
  }
  __syncthreads();
  return *s_fail == 0;
}

template <int BITS, int T>
__global__ void __launch_bounds__(kChThreads, 1) k_gemv_chain(const __grid_constant__ ChainParams P) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float s_red[kChWarps];
  __shared__ float s_r[T];
  __shared__ int s_fail;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * kChWarps + warp, nw = gridDim.x * kChWarps;
  const int d = P.st[0].cols;

  // a warp's units of a step: gw, gw + nw, ..., kChU of them requested at once
  RowGeo rg = row_geo(d, BITS);
  int rs = lane / rg.LPR, lp = lane - rs * rg.LPR;
  uint4 qv[kChU][kChNit];
  uint32_t sv[kChU][kChNit];
  auto load_batch = [&](const ChainStep& W, int ub) {
    const int units = (W.rows + rg.RPP - 1) / rg.RPP;
#pragma unroll
    for (int j = 0; j < kChU; ++j)
      if (ub + j * nw < units) ch_load<BITS>(W, rg, ub + j * nw, rs, lp, 0, qv[j], sv[j]);
  };
  // step 0's first rows, in flight during the norm and the staging
  load_batch(P.st[0], gw);

  // per-token norm factors, summed exactly as k_rmsnorm does (same thread count)
  if (P.norm) {
    for (int t = 0; t < T; ++t) {
      const uint16_t* xt = P.x + (size_t)t * d;
      float ss = 0.f;
      for (int i = threadIdx.x; i < d; i += kChThreads) {
        const float h = bf16f(xt[i]);
        ss = fmaf(h, h, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_red[warp] = ss;
      __syncthreads();
      if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int i = 0; i < kChWarps; ++i) tot += s_red[i];
        s_r[t] = 1.f / sqrtf(tot / (float)d + P.eps);
      }
      __syncthreads();
    }
  }

  for (int k = 0; k < P.n; ++k) {
    const ChainStep& W = P.st[k];
    const XStage st = xstage_carve(smem, T, W.cols);
    if (k == 0) {
      if (P.norm)
        stage_x24<BITS>(NormSrc{P.x, d, s_r, P.rho}, T, d, st);
      else
        stage_x24<BITS>(StridedSrc<uint16_t>{P.x, d}, T, d, st);
    } else {
      stage_x24<BITS>(ChainL2Src{P.buf[(k - 1) & 1], P.ldb}, T, W.cols, st);
    }
    const bool last = k == P.n - 1;
    const int units = (W.rows + rg.RPP - 1) / rg.RPP;
    // one token: this lane's parts of x, held in registers for the whole step
    // (up to kXr parts: 24 registers each at 4 bits, 48 at 2 bits)
    constexpr int kXr = T == 1 ? (BITS == 4 ? kChNit : 2) : 1;
    const bool xreg = T == 1 && rg.NIT <= kXr;
    uint4 xr_c[kXr][4 * Geo<BITS>::kNch];
    uint2 xr_h[kXr][4 * Geo<BITS>::kNch];
    float2 xr_p[kXr];
    if (xreg) {
#pragma unroll
      for (int i = 0; i < kXr; ++i)
        if (i < rg.NIT) {
          load_part_x<BITS>(st, 0, i, lp, rg, xr_c[i], xr_h[i]);
          xr_p[i] = st.partinfo[i * rg.LPR + lp];
        }
    }
    for (int ub = gw; ub < units; ub += kChU * nw) {
      if (ub != gw) load_batch(W, ub);  // the first batch was requested earlier
#pragma unroll
      for (int j = 0; j < kChU; ++j) {
        const int u = ub + j * nw;
        if (u >= units) break;
        if (xreg) {
          // one token: this lane's parts of x are the same for every row it
          // takes, so they were read from shared memory once (xr_* above)
          float a = 0.f;
#pragma unroll
          for (int i = 0; i < kXr; ++i)
            if (i < rg.NIT) a = part_dot_x<BITS>(qv[j][i], sv[j][i], xr_c[i], xr_h[i], xr_p[i], a);
          const float v = row_reduce(a, rg.LPR);
          const int row = u * rg.RPP + rs;
          if (lp == 0 && row < W.rows) {
            if (!last) {
              P.buf[k & 1][row] = f2bf(v);
            } else {
              const float y = P.residual ? bf16f(P.x[row]) + v : v;
              if (P.out) P.out[row] = f2bf(y);
              if (P.out_f32) P.out_f32[row] = y;
            }
          }
          continue;
        }
        float acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = 0.f;
        for (int it0 = 0; it0 < rg.NIT; it0 += kChNit) {
          uint4 qx[kChNit];
          uint32_t sx[kChNit];
          if (it0 > 0) ch_load<BITS>(W, rg, u, rs, lp, it0, qx, sx);  // rows wider than kChNit parts per lane
#pragma unroll
          for (int i = 0; i < kChNit; ++i) {
            const int it = it0 + i;
            if (it < rg.NIT) {
              const uint4 q = it0 > 0 ? qx[i] : qv[j][i];
              const uint32_t sw = it0 > 0 ? sx[i] : sv[j][i];
#pragma unroll
              for (int t = 0; t < T; ++t) acc[t] = part_dot24<BITS>(q, sw, st, t, it, lp, rg, acc[t]);
            }
          }
        }
        const int row = u * rg.RPP + rs;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float v = row_reduce(acc[t], rg.LPR);
          if (lp == 0 && row < W.rows) {
            if (!last) {
              P.buf[k & 1][(size_t)t * P.ldb + row] = f2bf(v);
            } else {
              const float y = P.residual ? bf16f(P.x[(size_t)t * d + row]) + v : v;
              if (P.out) P.out[(size_t)t * W.rows + row] = f2bf(y);
              if (P.out_f32) P.out_f32[(size_t)t * W.rows + row] = y;
            }
          }
        }
      }
    }
    if (last) break;
    // the next step's first rows, then the grid-wide wait for this step's outputs
    rg = row_geo(P.st[k + 1].cols, BITS);
    rs = lane / rg.LPR;
    lp = lane - rs * rg.LPR;
    load_batch(P.st[k + 1], gw);
    if (!ch_grid_wait(P, k, &s_fail)) return;
  }
}

size_t chain_smem_bytes(int max_cols, int bits, int T) { return xstage_bytes(T, max_cols, bits); }

template <int BITS, int T>
static cudaError_t launch_chain_t(const ChainParams& P, size_t sm, cudaStream_t s) {
  auto kern = k_gemv_chain<BITS, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kChThreads, sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  void* args[] = {const_cast<ChainParams*>(&P)};
  return cudaLaunchCooperativeKernel((void*)kern, dim3(num_sms()), dim3(kChThreads), args, sm, s);
}

template <int BITS>
static cudaError_t launch_chain_bits(const ChainParams& P, int T, size_t sm, cudaStream_t s) {
  switch (T) {
    case 1: return launch_chain_t<BITS, 1>(P, sm, s);
    case 2: return launch_chain_t<BITS, 2>(P, sm, s);
    case 3: return launch_chain_t<BITS, 3>(P, sm, s);
    case 4: return launch_chain_t<BITS, 4>(P, sm, s);
    case 5: return launch_chain_t<BITS, 5>(P, sm, s);
    case 6: return launch_chain_t<BITS, 6>(P, sm, s);
    case 7: return launch_chain_t<BITS, 7>(P, sm, s);
    default: return launch_chain_t<BITS, 8>(P, sm, s);
  }
}

cudaError_t launch_chain(const ChainStep* steps, int n, int bits, const uint16_t* x, int batch, int norm,
                         const uint16_t* rho, float eps, int residual, uint16_t* out, float* out_f32, Ctrl* ctrl,
                         int* counter, uint16_t* buf0, uint16_t* buf1, int ldb, long long timeout_ns, cudaStream_t s) {
  ChainParams P{};
  int max_cols = 0;
  for (int i = 0; i < n; ++i) {
    P.st[i] = steps[i];
    if (steps[i].cols > max_cols) max_cols = steps[i].cols;
  }
  P.n = n;
  P.x = x;
  P.norm = norm;
  P.rho = rho;
  P.eps = eps;
  P.residual = residual;
  P.out = out;
  P.out_f32 = out_f32;
  P.buf[0] = buf0;
  P.buf[1] = buf1;
  P.ldb = ldb;
  P.ctrl = ctrl;
  P.counter = counter;
  P.timeout_ns = timeout_ns;
  const size_t sm = chain_smem_bytes(max_cols, bits, batch);
  return bits == 4 ? launch_chain_bits<4>(P, batch, sm, s) : launch_chain_bits<2>(P, batch, sm, s);
}

}  // namespace bgq
