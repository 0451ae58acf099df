// gemv.cu — standalone group-quantized GEMV y = W x (bf16 out, fp32 accumulate).
//
// Flash-MoE page, section "FMA Dequant：一条指令省12%": every weight is
// nibble*scale + bias, and the product with x can be reordered into
// fma(nibble, scale*x, bias*x). Because scale and bias are constant over a
// group of 64 columns, the reordering summed over a group is
//     sum_k fma(q_k, s*x_k, b*x_k) = s * sum_k q_k x_k + b * sum_k x_k,
// so one multiply-add per weight remains (sum_k x_k is shared by all rows).
// The production kernel evaluates sum_k q_k x_k exactly in integers (dp4a on
// x held as 24-bit fixed point per group), which needs 0.75 dp4a per weight
// and keeps the GEMV memory-bound on GB300 at 4 and at 2 bits. The other
// three variants keep the per-weight floating-point forms for comparison.
//
// Work split: a CTA of 8 warps; each warp owns RPP rows (RPP = 32/LPR); the
// LPR lanes of a row each read one 16-byte part per iteration (split-K across
// lanes) and the partial sums meet in a shuffle reduction. x is staged once
// per CTA in shared memory. Row loads are issued before x is staged so their
// latency overlaps the staging.
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kMaxNit = 4;  // parts per lane held in registers at once

template <int BITS, int T>
__global__ void __launch_bounds__(kGemvThreads)
k_qgemv_int(const uint32_t* __restrict__ q, const uint32_t* __restrict__ sb, int rows, int cols,
              const uint16_t* __restrict__ x, int ldx, uint16_t* __restrict__ y, float* __restrict__ yf, int ldy,
              const uint16_t* __restrict__ res) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RowGeo rg = row_geo(cols, BITS);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rs = lane / rg.LPR, lp = lane - rs * rg.LPR;
  const int row = (blockIdx.x * kGemvWarps + warp) * rg.RPP + rs;
  const bool valid = row < rows;
  const int wpr = cols * BITS / 32, gpr = cols / kGroup;

  const XStage st = xstage_carve(smem, T, cols);

  const uint32_t* qrow = q + (size_t)(valid ? row : 0) * wpr;
  const uint32_t* sbrow = sb + (size_t)(valid ? row : 0) * gpr;

  uint4 qv[kMaxNit];
  uint32_t sv[kMaxNit];
  const int nfirst = rg.NIT < kMaxNit ? rg.NIT : kMaxNit;
#pragma unroll
  for (int i = 0; i < kMaxNit; ++i) {
    if (i < nfirst && valid) {
      int p = i * rg.LPR + lp;
      qv[i] = ldg_stream16(qrow + 4 * p);
      sv[i] = ldg_stream4(sbrow + part_group<BITS>(p));
    } else {
      qv[i] = make_uint4(0, 0, 0, 0);
      sv[i] = 0;
    }
  }

  pdl_wait();  // x may come from the previous kernel; y may still be read by it
  pdl_trigger();  // the next kernel may start its prologue now (at most one waits behind this one)
  stage_x24<BITS>(StridedSrc<uint16_t>{x, ldx}, T, cols, st);

  float acc[T];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t] = 0.f;

  for (int it0 = 0; it0 < rg.NIT; it0 += kMaxNit) {
    if (it0 > 0) {
#pragma unroll
      for (int i = 0; i < kMaxNit; ++i) {
        int it = it0 + i;
        if (it < rg.NIT && valid) {
          int p = it * rg.LPR + lp;
          qv[i] = ldg_stream16(qrow + 4 * p);
          sv[i] = ldg_stream4(sbrow + part_group<BITS>(p));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxNit; ++i) {
      int it = it0 + i;
      if (it < rg.NIT) {
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = part_dot24<BITS>(qv[i], sv[i], st, t, it, lp, rg, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < T; ++t) {
    float v = row_reduce(acc[t], rg.LPR);
    if (valid && lp == 0) {
      if (res) v += bf16f(res[(size_t)t * ldy + row]);  // a residual input: the fp32 sum, then one rounding
      if (y) y[(size_t)t * ldy + row] = f2bf(v);
      if (yf) yf[(size_t)t * ldy + row] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// Floating-point variants. x is staged as fp32 in the same lane-major slot
// order (word w of part p: its 32/BITS values in consecutive 16-byte slots).
// ---------------------------------------------------------------------------
template <int BITS>
__device__ void stage_x_f32(const uint16_t* __restrict__ x, int ldx, int T, int cols, float4* slots,
                            float* partsum) {
  using G = Geo<BITS>;
  const RowGeo rg = row_geo(cols, BITS);
  constexpr int NCH = G::kPer / 4;
  const int words = cols * BITS / 32;
  for (int tw = threadIdx.x; tw < T * words; tw += blockDim.x) {
    int t = tw / words, w = tw - t * words;
    int p = w >> 2, c = w & 3, it = p / rg.LPR, lp = p - it * rg.LPR;
    const uint16_t* xp = x + (size_t)t * ldx + w * G::kPer;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      float4 v = make_float4(bf16f(xp[4 * ch]), bf16f(xp[4 * ch + 1]), bf16f(xp[4 * ch + 2]), bf16f(xp[4 * ch + 3]));
      slots[(((t * rg.NIT + it) * 4 + c) * NCH + ch) * rg.LPR + lp] = v;
    }
  }
  // per-part sum of x (used by the hoisted variant)
  for (int tp = threadIdx.x; tp < T * rg.P; tp += blockDim.x) {
    int t = tp / rg.P, p = tp - t * rg.P;
    const uint16_t* xp = x + (size_t)t * ldx + p * G::kValsPerPart;
    float s = 0.f;
    for (int i = 0; i < G::kValsPerPart; ++i) s += bf16f(xp[i]);
    partsum[tp] = s;
  }
  __syncthreads();
}

template <int BITS, int VARIANT>
__global__ void __launch_bounds__(kGemvThreads)
k_qgemv_float(const uint32_t* __restrict__ q, const uint32_t* __restrict__ sb, int rows, int cols,
              const uint16_t* __restrict__ x, int ldx, int T, uint16_t* __restrict__ y, int ldy) {
  using G = Geo<BITS>;
  constexpr int NCH = G::kPer / 4;
  constexpr uint32_t mask = (1u << BITS) - 1u;
  extern __shared__ __align__(16) unsigned char smem[];
  const RowGeo rg = row_geo(cols, BITS);
  float4* slots = reinterpret_cast<float4*>(smem);
  float* partsum = reinterpret_cast<float*>(smem + (size_t)T * cols * 4);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rs = lane / rg.LPR, lp = lane - rs * rg.LPR;
  const int row = (blockIdx.x * kGemvWarps + warp) * rg.RPP + rs;
  const bool valid = row < rows;
  const int wpr = cols * BITS / 32, gpr = cols / kGroup;
  const uint32_t* qrow = q + (size_t)(valid ? row : 0) * wpr;
  const uint32_t* sbrow = sb + (size_t)(valid ? row : 0) * gpr;
  pdl_wait();
  pdl_trigger();
  stage_x_f32<BITS>(x, ldx, T, cols, slots, partsum);

  for (int t = 0; t < T; ++t) {
    float acc = 0.f;
    for (int it = 0; it < rg.NIT; ++it) {
      int p = it * rg.LPR + lp;
      uint4 qv = valid ? ldg_stream16(qrow + 4 * p) : make_uint4(0, 0, 0, 0);
      uint32_t sbw = valid ? ldg_stream4(sbrow + part_group<BITS>(p)) : 0u;
      float s = bf16lo(sbw), b = bf16hi(sbw);
      const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
      float aq = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          float4 xv = slots[(((t * rg.NIT + it) * 4 + c) * NCH + ch) * rg.LPR + lp];
          const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float qf = __uint2float_rn((qw[c] >> (BITS * (4 * ch + i))) & mask);
            if (VARIANT == 1) {  // standard: (q*s + b) * x
              acc = fmaf(fmaf(qf, s, b), xs[i], acc);
            } else if (VARIANT == 2) {  // reordered: fma(q, s*x, b*x)
              acc += fmaf(qf, s * xs[i], b * xs[i]);
            } else {  // hoisted over the group part
              aq = fmaf(qf, xs[i], aq);
            }
          }
        }
      }
      if (VARIANT == 3) acc = fmaf(s, aq, fmaf(b, partsum[t * rg.P + p], acc));
    }
    float v = row_reduce(acc, rg.LPR);
    if (valid && lp == 0) y[(size_t)t * ldy + row] = f2bf(v);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
size_t qgemv_int_smem(int cols, int bits, int T) { return xstage_bytes(T, cols, bits); }

template <int BITS, int T>
static cudaError_t launch_int_t(const QMat& W, const uint16_t* x, int ldx, uint16_t* y, float* yf, int ldy,
                                  const uint16_t* res, cudaStream_t s) {
  RowGeo rg = row_geo(W.cols, BITS);
  int rows_per_cta = kGemvWarps * rg.RPP;
  int grid = (W.rows + rows_per_cta - 1) / rows_per_cta;
  size_t sm = qgemv_int_smem(W.cols, BITS, T);
  auto kern = k_qgemv_int<BITS, T>;
  if (sm > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  return launch_overlapped(kern, grid, kGemvThreads, sm, s, W.q, reinterpret_cast<const uint32_t*>(W.sb), W.rows,
                           W.cols, x, ldx, y, yf, ldy, res);
}

template <int BITS>
static cudaError_t launch_int_bits(const QMat& W, const uint16_t* x, int ldx, uint16_t* y, float* yf, int ldy,
                                     const uint16_t* res, int T, cudaStream_t s) {
  switch (T) {
    case 1: return launch_int_t<BITS, 1>(W, x, ldx, y, yf, ldy, res, s);
    case 2: return launch_int_t<BITS, 2>(W, x, ldx, y, yf, ldy, res, s);
    case 3: return launch_int_t<BITS, 3>(W, x, ldx, y, yf, ldy, res, s);
    case 4: return launch_int_t<BITS, 4>(W, x, ldx, y, yf, ldy, res, s);
    case 5: return launch_int_t<BITS, 5>(W, x, ldx, y, yf, ldy, res, s);
    case 6: return launch_int_t<BITS, 6>(W, x, ldx, y, yf, ldy, res, s);
    case 7: return launch_int_t<BITS, 7>(W, x, ldx, y, yf, ldy, res, s);
    default: return launch_int_t<BITS, 8>(W, x, ldx, y, yf, ldy, res, s);
  }
}

// Inputs staged per launch of the integer kernel: up to 8, as many as fit in
// the 227 KB of shared memory of a CTA.
static int qgemv_max_tokens(int cols, int bits) {
  const size_t per = xstage_bytes(1, cols, bits);
  const int n = (int)((size_t)227 * 1024 / per);
  return n < 8 ? n : 8;
}

cudaError_t launch_qgemv(const QMat& W, const uint16_t* x, int batch, uint16_t* y, float* yf, int variant,
                         cudaStream_t s, const uint16_t* res) {
  const int tmax = variant == 0 ? qgemv_max_tokens(W.cols, W.bits) : 8;
  if (tmax < 1 || (res && variant != 0)) return cudaErrorInvalidValue;
  for (int t0 = 0; t0 < batch; t0 += tmax) {
    int T = batch - t0 < tmax ? batch - t0 : tmax;
    const uint16_t* xt = x + (size_t)t0 * W.cols;
    uint16_t* yt = y ? y + (size_t)t0 * W.rows : nullptr;
    float* yft = yf ? yf + (size_t)t0 * W.rows : nullptr;
    const uint16_t* rt = res ? res + (size_t)t0 * W.rows : nullptr;
    cudaError_t e;
    if (variant == 0) {
      e = W.bits == 4 ? launch_int_bits<4>(W, xt, W.cols, yt, yft, W.rows, rt, T, s)
                      : launch_int_bits<2>(W, xt, W.cols, yt, yft, W.rows, rt, T, s);
    } else {
      RowGeo rg = row_geo(W.cols, W.bits);
      int rows_per_cta = kGemvWarps * rg.RPP;
      int grid = (W.rows + rows_per_cta - 1) / rows_per_cta;
      size_t sm = (size_t)T * W.cols * 4 + (size_t)T * rg.P * 4;
      void (*kern)(const uint32_t*, const uint32_t*, int, int, const uint16_t*, int, int, uint16_t*, int) = nullptr;
      if (W.bits == 4) {
        kern = variant == 1 ? k_qgemv_float<4, 1> : variant == 2 ? k_qgemv_float<4, 2> : k_qgemv_float<4, 3>;
      } else {
        kern = variant == 1 ? k_qgemv_float<2, 1> : variant == 2 ? k_qgemv_float<2, 2> : k_qgemv_float<2, 3>;
      }
      if (sm > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
      }
      e = launch_overlapped(kern, grid, kGemvThreads, sm, s, W.q, reinterpret_cast<const uint32_t*>(W.sb), W.rows,
                            W.cols, xt, W.cols, T, yt, W.rows);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bgq
