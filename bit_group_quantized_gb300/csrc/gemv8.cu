// gemv8.cu — 8-bit group-quantized GEMV y = W x (bf16 out, fp32 accumulate):
// the int8 weight format of dense MLP and QKV projections.
//
// Source: "Redis 之父下场手写推理引擎：antirez 用约 24000 行原生代码驯服视频生成模型"
// (text-matrix.pages.dev), the paragraph on --use-int8-row-fc2: the engine's
// default MLP weights are int8 with one scale per group, QKV projections were
// quantised the same way afterwards, and the option swaps the MLP's second
// fully connected layer (FC2) for int8 with a single scale per row.
// Readings: the format is this library's affine one at 8 bits, codes q in
// 0..255 (four per uint32, least-significant byte first), W = q*s + b with a
// bf16 (scale, bias) pair per group of 64 columns, or one pair per row for the
// per-row variant. Symmetric signed int8 (W = c*s, c in -128..127) is the
// special case q = c + 128, b = -128*s, exact in bf16.
//
// Dot product: the same group reordering as the 4-bit kernels (Flash-MoE page,
// "FMA Dequant"): per 16-code part, y += s*2^-sh*sum(q*X) + b*2^-sh*sum(X),
// with x held as 24-bit fixed point X (one power-of-two exponent 2^-sh per
// group of 64 inputs) split into two unsigned bytes and a signed high byte.
// Codes are whole bytes, so each word of 4 codes needs three dp4a and no
// masking: 0.75 dp4a per weight and token, as at 4 bits.
//
// Work split: 8 warps per CTA; the LPR lanes of a row each read one 16-byte
// part (16 codes) per iteration, up to 8 parts in flight per lane; partial sums
// meet in a shuffle reduction. Inputs are staged once per CTA in shared memory
// in lane-major order (the lanes of a row read consecutive 16-byte slots).
// One or two inputs: one row per warp, the whole matrix requested at once
// (k_q8gemv); three to eight: a persistent grid whose warps stream their rows
// with the next rows in flight, so the inputs are staged once per CTA rather
// than once per 8 rows (k_q8gemv_stream).
// The kernel is launched overlapped with the previous kernel on the stream
// (programmatic dependent launch): its weight loads start before that kernel
// has finished, and it waits for it only before reading x.
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kG8Threads = 256;
constexpr int kG8Warps = kG8Threads / 32;
constexpr int kG8Nit = 8;  // parts per lane held in registers at once
constexpr int kG8MaxSmem = 227 * 1024;  // dynamic shared memory per CTA on sm_103a

// Shared-memory bytes for T staged inputs of `cols` values: 3 bytes of X per
// value (L, M, H bytes) plus (2^-sh, 2^-sh * sum X) per 16-value part.
__host__ __device__ inline size_t q8_stage_bytes(int cols, int T) {
  return (size_t)T * cols * 3 + (size_t)T * (cols / 16) * 8;
}

// Stage T inputs, one thread per 8 values (two code words). Slot of part p,
// half j of token t: ((t*NIT + p/LPR)*2 + j)*LPR + p%LPR holds
// {L(word 2j), M(word 2j), L(word 2j+1), M(word 2j+1)} in `slots` and
// {H(word 2j), H(word 2j+1)} in `hslots`, byte i of L/M/H belonging to code i
// of that word. Each thread first requests up to AHEAD
// of its 16-byte input pieces, then converts them, so one load latency is paid
// per AHEAD passes. All threads of the block call; ends with __syncthreads().
template <int AHEAD>
__device__ void stage_x8(const uint16_t* __restrict__ x, int ldx, int T, int cols, const RowGeo rg,
                         uint4* __restrict__ slots, uint2* __restrict__ hslots, float2* __restrict__ partinfo) {
  const int hpr = cols / 8;  // 8-value halves of a part per token (a multiple of 8)
  const int total = T * hpr;
  // t = floor(i / hpr); with many passes through a float reciprocal, exact
  // while total < 2^20 (the fraction of (i + 0.5) / hpr stays >= 0.5 / hpr
  // away from an integer); with few, the integer division needs fewer registers
  const float inv_hpr = 1.f / (float)hpr;
  auto token_of = [&](int i) { return AHEAD <= 2 ? i / hpr : (int)(((float)i + 0.5f) * inv_hpr); };
  for (int base = 0; base < total; base += AHEAD * blockDim.x) {
    uint4 raw[AHEAD];
#pragma unroll
    for (int r = 0; r < AHEAD; ++r) {
      const int i = base + r * blockDim.x + threadIdx.x;
      if (i < total) {
        const int t = token_of(i), h = i - t * hpr;
        raw[r] = *reinterpret_cast<const uint4*>(x + (size_t)t * ldx + 8 * h);
      } else {
        raw[r] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int r = 0; r < AHEAD; ++r) {
      // uniform trip count: every lane reaches the shuffles; a group of 64
      // values is 8 consecutive, aligned lanes (hpr and blockDim are multiples of 8)
      const int i = base + r * blockDim.x + threadIdx.x;
      const bool active = i < total;
      const int t = active ? token_of(i) : 0;
      const int h = active ? i - t * hpr : 0;
      float v[8];
      unpack_bf16x8(raw[r], v);
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      const int sh = x24_shift(m);
      const float sc = exp2i(sh);
      int X[8];
      int xsum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        X[k] = x24_fix(v[k], sc);
        xsum += X[k];
      }
      uint32_t L0, M0, H0, L1, M1, H1;
      pack24(X[0], X[1], X[2], X[3], L0, M0, H0);
      pack24(X[4], X[5], X[6], X[7], L1, M1, H1);
      const int p = h >> 1, j = h & 1;
      const int it = p / rg.LPR, lp = p - it * rg.LPR;
      if (active) {
        const int slot = ((t * rg.NIT + it) * 2 + j) * rg.LPR + lp;
        slots[slot] = make_uint4(L0, M0, L1, M1);
        hslots[slot] = make_uint2(H0, H1);
      }
      xsum += __shfl_xor_sync(kFull, xsum, 1);  // the part's other half
      if (active && j == 0) {
        const float inv = exp2i(-sh);
        partinfo[t * rg.P + p] = make_float2(inv, (float)xsum * inv);
      }
    }
  }
  __syncthreads();
}

// sum over the part of q*s + b times x, added to acc (see the file comment).
// SPLIT: four independent dp4a chains (two deep) instead of two (four deep);
// used where T tokens give the registers room (the chains' latency is the
// main stall there), while the single-token kernel stays within 64 registers.
template <bool SPLIT>
__device__ __forceinline__ float part_dot8(const uint4 qv, uint32_t sbw, const uint4 x0, const uint4 x1,
                                           const uint2 h0v, const uint2 h1v, const float2 pi, float acc) {
  int lo, hi;
  if (SPLIT) {
    uint32_t l0 = dp4a_uu(qv.x, x0.x, 0u), l1 = dp4a_uu(qv.y, x0.z, 0u);
    uint32_t m0 = dp4a_uu(qv.x, x0.y, 0u), m1 = dp4a_uu(qv.y, x0.w, 0u);
    int h0 = dp4a_us(qv.x, h0v.x, 0), h1 = dp4a_us(qv.y, h0v.y, 0);
    l0 = dp4a_uu(qv.z, x1.x, l0);
    l1 = dp4a_uu(qv.w, x1.z, l1);
    m0 = dp4a_uu(qv.z, x1.y, m0);
    m1 = dp4a_uu(qv.w, x1.w, m1);
    h0 = dp4a_us(qv.z, h1v.x, h0);
    h1 = dp4a_us(qv.w, h1v.y, h1);
    lo = (int)(l0 + l1) + (int)(m0 + m1) * 256;  // < 16*255*255*257 < 2^31
    hi = h0 + h1;
  } else {
    uint32_t l = dp4a_uu(qv.x, x0.x, 0u), m = dp4a_uu(qv.x, x0.y, 0u);
    int h = dp4a_us(qv.x, h0v.x, 0);
    l = dp4a_uu(qv.y, x0.z, l);
    m = dp4a_uu(qv.y, x0.w, m);
    h = dp4a_us(qv.y, h0v.y, h);
    l = dp4a_uu(qv.z, x1.x, l);
    m = dp4a_uu(qv.z, x1.y, m);
    h = dp4a_us(qv.z, h1v.x, h);
    l = dp4a_uu(qv.w, x1.z, l);
    m = dp4a_uu(qv.w, x1.w, m);
    h = dp4a_us(qv.w, h1v.y, h);
    lo = (int)l + (int)m * 256;
    hi = h;
  }
  const float A = fmaf((float)hi, 65536.f, (float)lo);
  const float s = bf16lo(sbw), b = bf16hi(sbw);
  return fmaf(s * pi.x, A, fmaf(b, pi.y, acc));
}

// gpr = (scale, bias) pairs per row: cols/64, or 1 for the per-row format.
template <int T>
__global__ void __launch_bounds__(kG8Threads, T <= 2 ? 4 : 3)
k_q8gemv(const uint32_t* __restrict__ q, const uint32_t* __restrict__ sb, int rows, int cols, int gpr,
         const uint16_t* __restrict__ x, int ldx, uint16_t* __restrict__ y, int ldy) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RowGeo rg = row_geo(cols, 8);
  uint4* slots = reinterpret_cast<uint4*>(smem);
  uint2* hslots = reinterpret_cast<uint2*>(smem + (size_t)T * cols * 2);
  float2* partinfo = reinterpret_cast<float2*>(smem + (size_t)T * cols * 3);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rs = lane / rg.LPR, lp = lane - rs * rg.LPR;
  const int row = (blockIdx.x * kG8Warps + warp) * rg.RPP + rs;
  const bool valid = row < rows;
  const int wpr = cols / 4;
  const bool per_row = gpr == 1;
  const uint32_t* qrow = q + (size_t)(valid ? row : 0) * wpr;
  const uint32_t* sbrow = sb + (size_t)(valid ? row : 0) * gpr;

  // the row's first parts are requested before the inputs are staged (and
  // before the previous kernel on the stream has finished)
  uint4 qv[kG8Nit];
  uint32_t sv[kG8Nit];
#pragma unroll
  for (int i = 0; i < kG8Nit; ++i) {
    const int p = i * rg.LPR + lp;
    if (i < rg.NIT && valid) {
      qv[i] = ldg_stream16(qrow + 4 * p);
      sv[i] = ldg_stream4(sbrow + (per_row ? 0 : (p >> 2)));
    } else {
      qv[i] = make_uint4(0, 0, 0, 0);
      sv[i] = 0;
    }
  }

  pdl_wait();  // x may come from the previous kernel; y may still be read by it
  pdl_trigger();  // the next kernel may start its prologue now (at most one waits behind this one)
  stage_x8<T <= 2 ? 2 : 4>(x, ldx, T, cols, rg, slots, hslots, partinfo);

  float acc[T];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t] = 0.f;
  for (int it0 = 0; it0 < rg.NIT; it0 += kG8Nit) {
    if (it0 > 0) {
#pragma unroll
      for (int i = 0; i < kG8Nit; ++i) {
        const int it = it0 + i, p = it * rg.LPR + lp;
        if (it < rg.NIT && valid) {
          qv[i] = ldg_stream16(qrow + 4 * p);
          sv[i] = ldg_stream4(sbrow + (per_row ? 0 : (p >> 2)));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kG8Nit; ++i) {
      const int it = it0 + i;
      if (it < rg.NIT) {
        const size_t xs = (size_t)(it * 2) * rg.LPR + lp;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const size_t xt = xs + (size_t)t * rg.NIT * 2 * rg.LPR;
          acc[t] = part_dot8<(T >= 3)>(qv[i], sv[i], slots[xt], slots[xt + rg.LPR], hslots[xt], hslots[xt + rg.LPR],
                                       partinfo[t * rg.P + it * rg.LPR + lp], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const float v = row_reduce(acc[t], rg.LPR);
    if (valid && lp == 0) y[(size_t)t * ldy + row] = f2bf(v);
  }
}

// One warp's work items. A warp owns row groups gw, gw + W, ... (W = warps in
// the grid; a row group is RPP rows, one per LPR lanes). An item fills the
// lanes' kG8Nit part registers: RI = kG8Nit / NIT row groups whole when a row
// has fewer parts per lane (NIT dividing kG8Nit), else one chunk of up to
// kG8Nit parts of one row group (nchunk chunks per row group).
struct Q8Item {
  const uint32_t* q;
  const uint32_t* sb;
  int rows, wpr, gpr, gw, W, nchunk, RI, nmine;
  RowGeo rg;
  int rs, lp;
  // part slot i of item `item`: local row group j (of this warp), part index it
  __device__ __forceinline__ void slot(int item, int i, int& j, int& it) const {
    if (RI == 1) {
      j = item / nchunk;
      it = (item - j * nchunk) * kG8Nit + i;
    } else {
      const int r = i / rg.NIT;
      j = item * RI + r;
      it = i - r * rg.NIT;
    }
  }
  __device__ __forceinline__ int row_of(int j) const { return (gw + j * W) * rg.RPP + rs; }
  __device__ __forceinline__ bool live(int j, int it) const { return j < nmine && it < rg.NIT; }
  __device__ __forceinline__ void load(int item, uint4 (&qv)[kG8Nit], uint32_t (&sv)[kG8Nit]) const {
#pragma unroll
    for (int i = 0; i < kG8Nit; ++i) {
      int j, it;
      slot(item, i, j, it);
      const int row = row_of(j), p = it * rg.LPR + lp;
      if (live(j, it) && row < rows) {
        qv[i] = ldg_stream16(q + (size_t)row * wpr + 4 * p);
        sv[i] = ldg_stream4(sb + (size_t)row * gpr + (gpr == 1 ? 0 : (p >> 2)));
      } else {
        qv[i] = make_uint4(0, 0, 0, 0);
        sv[i] = 0;
      }
    }
  }
};

// Dot products of one item with the T staged inputs; after a row group's last
// part its sums are reduced over the row's lanes, stored, and reset.
template <int T>
__device__ __forceinline__ void q8_item(const Q8Item& I, int item, const uint4 (&qv)[kG8Nit],
                                        const uint32_t (&sv)[kG8Nit], const uint4* slots, const uint2* hslots,
                                        const float2* partinfo,
                                        float (&acc)[T], uint16_t* __restrict__ y, int ldy) {
  const RowGeo& rg = I.rg;
#pragma unroll
  for (int i = 0; i < kG8Nit; ++i) {
    int j, it;
    I.slot(item, i, j, it);
    if (I.live(j, it)) {
      const size_t xs = (size_t)(it * 2) * rg.LPR + I.lp;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const size_t xt = xs + (size_t)t * rg.NIT * 2 * rg.LPR;
        acc[t] = part_dot8<(T >= 3)>(qv[i], sv[i], slots[xt], slots[xt + rg.LPR], hslots[xt], hslots[xt + rg.LPR],
                                     partinfo[t * rg.P + it * rg.LPR + I.lp], acc[t]);
      }
      if (it == rg.NIT - 1) {  // warp-uniform
        const int row = I.row_of(j);
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float v = row_reduce(acc[t], rg.LPR);
          if (row < I.rows && I.lp == 0) y[(size_t)t * ldy + row] = f2bf(v);
          acc[t] = 0.f;
        }
      }
    }
  }
}

// Persistent streaming GEMV for 3..8 inputs: at most two CTAs per SM (the
// register limit), each warp walks its items with the next item's weights in
// flight while it computes the current one (two register buffers: up to 8 KB
// per warp, 128 KB per SM in flight). The inputs are staged once per CTA
// instead of once per 8 rows: at 4096 x 4096 this takes batch 4 from 16.2 to
// 13.2 us and batch 8 from 29.7 to 23.4 us, while at batch 1 the one-shot
// kernel above, which requests the whole matrix at once, stays faster
// (6.5 vs 6.9 us; 16384 x 4096: 17.7 vs 25.1 us; same box, same run).
// gpr = (scale, bias) pairs per row: cols/64, or 1 for the per-row format.
template <int T>
__global__ void __launch_bounds__(kG8Threads, 2)
k_q8gemv_stream(const uint32_t* __restrict__ q, const uint32_t* __restrict__ sb, int rows, int cols, int gpr,
         const uint16_t* __restrict__ x, int ldx, uint16_t* __restrict__ y, int ldy) {
  extern __shared__ __align__(16) unsigned char smem[];
  Q8Item I;
  I.rg = row_geo(cols, 8);
  uint4* slots = reinterpret_cast<uint4*>(smem);
  uint2* hslots = reinterpret_cast<uint2*>(smem + (size_t)T * cols * 2);
  float2* partinfo = reinterpret_cast<float2*>(smem + (size_t)T * cols * 3);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  I.rs = lane / I.rg.LPR;
  I.lp = lane - I.rs * I.rg.LPR;
  I.q = q;
  I.sb = sb;
  I.rows = rows;
  I.wpr = cols / 4;
  I.gpr = gpr;
  I.W = gridDim.x * kG8Warps;
  I.gw = blockIdx.x * kG8Warps + warp;
  const bool pack = I.rg.NIT < kG8Nit && kG8Nit % I.rg.NIT == 0;
  I.RI = pack ? kG8Nit / I.rg.NIT : 1;
  I.nchunk = pack ? 1 : (I.rg.NIT + kG8Nit - 1) / kG8Nit;
  const int nrg = (rows + I.rg.RPP - 1) / I.rg.RPP;
  I.nmine = I.gw < nrg ? (nrg - 1 - I.gw) / I.W + 1 : 0;
  const int nitems = pack ? (I.nmine + I.RI - 1) / I.RI : I.nmine * I.nchunk;

  // the first two items' weights are requested before the inputs are staged
  // (and before the previous kernel on the stream has finished)
  uint4 qa[kG8Nit], qb[kG8Nit];
  uint32_t sa[kG8Nit], sbv[kG8Nit];
  if (nitems > 0) I.load(0, qa, sa);
  if (nitems > 1) I.load(1, qb, sbv);

  pdl_wait();  // x may come from the previous kernel; y may still be read by it
  pdl_trigger();  // the next kernel may start its prologue now (at most one waits behind this one)
  stage_x8<T <= 2 ? 2 : 4>(x, ldx, T, cols, I.rg, slots, hslots, partinfo);

  float acc[T];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t] = 0.f;
  for (int item = 0; item < nitems; item += 2) {
    q8_item<T>(I, item, qa, sa, slots, hslots, partinfo, acc, y, ldy);
    if (item + 2 < nitems) I.load(item + 2, qa, sa);
    if (item + 1 < nitems) {
      q8_item<T>(I, item + 1, qb, sbv, slots, hslots, partinfo, acc, y, ldy);
      if (item + 3 < nitems) I.load(item + 3, qb, sbv);
    }
  }
}

// Largest number of inputs staged per launch for `cols` columns (0: too wide).
int q8gemv_max_tokens(int cols) {
  int T = 8;
  while (T > 0 && q8_stage_bytes(cols, T) > (size_t)kG8MaxSmem) --T;
  return T;
}

template <int T>
static cudaError_t launch_q8_t(const QMat& W, int gpr, const uint16_t* x, uint16_t* y, int ldy, cudaStream_t s) {
  const RowGeo rg = row_geo(W.cols, 8);
  const size_t sm = q8_stage_bytes(W.cols, T);
  int grid;
  void (*kern)(const uint32_t*, const uint32_t*, int, int, int, const uint16_t*, int, uint16_t*, int);
  if (T <= 2) {  // one-shot: 8 rows per CTA, the whole matrix requested at once
    const int rows_per_cta = kG8Warps * rg.RPP;
    grid = (W.rows + rows_per_cta - 1) / rows_per_cta;
    kern = k_q8gemv<T <= 2 ? T : 1>;
  } else {  // persistent: at most two CTAs per SM
    const int nrg = (W.rows + rg.RPP - 1) / rg.RPP;  // one warp's row groups
    int dev = 0, nsm = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e0 != cudaSuccess) return e0;
    grid = (nrg + kG8Warps - 1) / kG8Warps;
    if (grid > 2 * nsm) grid = 2 * nsm;
    kern = k_q8gemv_stream<T >= 3 ? T : 3>;
  }
  if (sm > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  return launch_overlapped(kern, grid, kG8Threads, sm, s, W.q, reinterpret_cast<const uint32_t*>(W.sb), W.rows,
                           W.cols, gpr, x, W.cols, y, ldy);
}

cudaError_t launch_q8gemv(const QMat& W, int gpr, const uint16_t* x, int batch, uint16_t* y, cudaStream_t s) {
  const int tmax = q8gemv_max_tokens(W.cols);
  if (tmax < 1) return cudaErrorInvalidValue;
  for (int t0 = 0; t0 < batch; t0 += tmax) {
    const int T = batch - t0 < tmax ? batch - t0 : tmax;
    const uint16_t* xt = x + (size_t)t0 * W.cols;
    uint16_t* yt = y + (size_t)t0 * W.rows;
    cudaError_t e;
    switch (T) {
      case 1: e = launch_q8_t<1>(W, gpr, xt, yt, W.rows, s); break;
      case 2: e = launch_q8_t<2>(W, gpr, xt, yt, W.rows, s); break;
      case 3: e = launch_q8_t<3>(W, gpr, xt, yt, W.rows, s); break;
      case 4: e = launch_q8_t<4>(W, gpr, xt, yt, W.rows, s); break;
      case 5: e = launch_q8_t<5>(W, gpr, xt, yt, W.rows, s); break;
      case 6: e = launch_q8_t<6>(W, gpr, xt, yt, W.rows, s); break;
      case 7: e = launch_q8_t<7>(W, gpr, xt, yt, W.rows, s); break;
      default: e = launch_q8_t<8>(W, gpr, xt, yt, W.rows, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bgq
