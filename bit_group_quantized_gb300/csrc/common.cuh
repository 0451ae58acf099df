// common.cuh — device helpers shared by the libbgq kernels.
//
// Packed format (Flash-MoE page, "FMA Dequant": w = nibble*scale + bias):
//   codes  uint32 [rows][cols*BITS/32], column k at word k/(32/BITS), bit offset BITS*(k%(32/BITS));
//   sb     bf16 pairs [rows][cols/64][2] = (scale, bias) per group of 64 columns.
//
// A row is consumed in "parts" of 128 bits of codes (one 16-byte load per lane):
// 32 columns at 4 bits (half a group), 64 columns at 2 bits (one group).
// P = cols*BITS/128 parts per row. A warp gives LPR = min(P, 32) lanes to a row,
// so it covers RPP = 32/LPR rows at once, each in NIT = P/LPR iterations.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bgq {

constexpr int kGroup = 64;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf16f(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// 4-way byte dot products (dp4a): unsigned codes times signed / unsigned bytes.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Streaming 16-byte / 4-byte global loads that do not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

template <int BITS>
struct Geo {
  static constexpr int kPer = 32 / BITS;         // codes per word
  static constexpr int kNvec = kPer / 4;         // byte vectors per word (4 codes each)
  static constexpr int kNch = kNvec / 2;         // staged x chunks per word (2 byte vectors each)
  static constexpr int kValsPerPart = 128 / BITS;
  static constexpr uint32_t kByteMask = BITS == 4 ? 0x0f0f0f0fu : 0x03030303u;
};

// Runtime row geometry for a given column count.
struct RowGeo {
  int P;    // parts per row
  int LPR;  // lanes per row
  int RPP;  // rows per warp pass
  int NIT;  // iterations per row
};
__host__ __device__ inline RowGeo row_geo(int cols, int bits) {
  RowGeo g;
  g.P = cols * bits / 128;
  g.LPR = g.P >= 32 ? 32 : g.P;
  g.RPP = 32 / g.LPR;
  g.NIT = g.P / g.LPR;
  return g;
}
__host__ __device__ inline bool cols_supported(int cols, int bits) {
  if (cols <= 0 || cols % kGroup) return false;
  int P = cols * bits / 128;
  if (P <= 0) return false;
  return (P % 32 == 0) || (32 % P == 0);
}

// ---------------------------------------------------------------------------
// x staging for the integer (dp4a) dot product.
//
// Per group of 64 inputs: sh = 22 - floor(log2(max|x|)), X_k = rn(x_k * 2^sh),
// so |X_k| < 2^23: 24-bit fixed point with one power-of-two exponent per
// group. Every bf16 input within 2^15 of its group's maximum is exact, and
// an fp32 input keeps 23 bits below the group maximum (an fp32 dot product's
// own rounding is 2^-24 of its terms). X is split into three bytes,
// X = 65536*H + 256*M + L (L, M unsigned, H signed), and each code byte
// vector meets them in three dp4a: 0.75 dp4a per weight and token.
// For code word w and byte vector j (codes k = w*per + j + nvec*i, i = 0..3)
// the L, M and H bytes of those four inputs form three uint32. Chunk ch of
// word w holds vectors 2ch, 2ch+1: {L0, M0, L1, M1} in the 16-byte array
// `chunks` and {H0, H1} in the 8-byte array `hib`, both at slot
//   (((t*NIT + p/LPR)*4 + c)*NCH + ch)*LPR + p%LPR
// (part p, word c of the part), so that for fixed (t, iteration, c, ch) the
// lanes of a row read consecutive slots (no bank conflicts). Part info
// (2^-sh, 2^-sh * sum_k X_k) is a float2 at [t*P + p].
// ---------------------------------------------------------------------------
struct XStage {
  uint4* chunks;    // [T * P * 4 * NCH] 16-byte slots (L, M bytes)
  uint2* hib;       // [T * P * 4 * NCH] 8-byte slots (H bytes)
  float2* partinfo; // [T * P]
};

// Bytes of T staged inputs of `cols` values: 3 bytes per value, 8 per part.
__host__ __device__ inline size_t xstage_bytes(int T, int cols, int bits) {
  return (size_t)T * cols * 3 + (size_t)T * (cols * bits / 128) * 8;
}
// The staging arrays of T inputs of `cols` values, carved from `base` (16-byte aligned).
__host__ __device__ inline XStage xstage_carve(void* base, int T, int cols) {
  XStage s;
  unsigned char* b = static_cast<unsigned char*>(base);
  s.chunks = reinterpret_cast<uint4*>(b);
  s.hib = reinterpret_cast<uint2*>(b + (size_t)T * cols * 2);
  s.partinfo = reinterpret_cast<float2*>(b + (size_t)T * cols * 3);
  return s;
}

// Input element loaders.
__device__ __forceinline__ float load_in(const uint16_t* x, int i) { return bf16f(x[i]); }
__device__ __forceinline__ float load_in(const float* x, int i) { return x[i]; }

// Where the T input vectors of a staging call come from. load8(t, k0, v)
// reads values k0..k0+7 of vector t (k0 a multiple of 8).
__device__ __forceinline__ void unpack_bf16x8(const uint4 u, float* v) {
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}
__device__ __forceinline__ void load8_from(const uint16_t* p, float* v) {
  unpack_bf16x8(*reinterpret_cast<const uint4*>(p), v);
}
__device__ __forceinline__ void load8_from(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <typename In>
struct StridedSrc {  // token t at x + t*ld (16-byte aligned rows)
  const In* x;
  int ld;
  __device__ void load8(int t, int k0, float* v) const { load8_from(x + (size_t)t * ld + k0, v); }
};
template <typename In>
struct GatherSrc {  // token t at base + off[t] (off in shared memory)
  const In* base;
  const int* off;
  __device__ void load8(int t, int k0, float* v) const { load8_from(base + off[t] + k0, v); }
};

// The shift sh = 22 - floor(log2 m) of a group whose largest magnitude is m
// (0 for an all-zero group), kept within [-126, 126] so that 2^sh and 2^-sh
// are normal floats.
__device__ __forceinline__ int x24_shift(float m) {
  if (!(m > 0.f)) return 0;
  const int e = (int)((__float_as_uint(m) >> 23) & 0xff) - 127;  // floor(log2 m) for normal m
  const int sh = 22 - e;
  return sh > 126 ? 126 : (sh < -126 ? -126 : sh);
}
// rn(v * 2^sh) for |v * 2^sh| < 2^23 (the product is exact). Rounding can
// only reach +2^23 (a value within half a unit below it); it is kept at
// 2^23 - 1. -2^23 is representable as (H, M, L) = (-128, 0, 0).
__device__ __forceinline__ int x24_fix(float v, float sc) { return min(__float2int_rn(v * sc), 8388607); }

// The L, M and H bytes of four 24-bit values (byte i from x_i).
__device__ __forceinline__ void pack24(int x0, int x1, int x2, int x3, uint32_t& L, uint32_t& M, uint32_t& H) {
  const uint32_t t01 = __byte_perm((uint32_t)x0, (uint32_t)x1, 0x5140);  // x0.b0 x1.b0 x0.b1 x1.b1
  const uint32_t t23 = __byte_perm((uint32_t)x2, (uint32_t)x3, 0x5140);
  L = __byte_perm(t01, t23, 0x5410);
  M = __byte_perm(t01, t23, 0x7632);
  const uint32_t u01 = __byte_perm((uint32_t)x0, (uint32_t)x1, 0x0062);  // x0.b2 x1.b2
  const uint32_t u23 = __byte_perm((uint32_t)x2, (uint32_t)x3, 0x0062);
  H = __byte_perm(u01, u23, 0x5410);
}

// Store the staged bytes of code word w (part p = w/4, word c = w%4) of token t.
template <int BITS>
__device__ __forceinline__ void store_word24(const int (&X)[Geo<BITS>::kPer], int t, int w, const RowGeo& rg,
                                             int lpr_shift, const XStage& st) {
  using G = Geo<BITS>;
  uint32_t L[G::kNvec], M[G::kNvec], H[G::kNvec];
#pragma unroll
  for (int j = 0; j < G::kNvec; ++j)
    pack24(X[j], X[j + G::kNvec], X[j + 2 * G::kNvec], X[j + 3 * G::kNvec], L[j], M[j], H[j]);
  const int p = w >> 2, c = w & 3;
  const int it = p >> lpr_shift, lp = p & (rg.LPR - 1);
  const int slot = ((((t * rg.NIT + it) * 4 + c) * G::kNch) << lpr_shift) + lp;
#pragma unroll
  for (int ch = 0; ch < G::kNch; ++ch) {
    st.chunks[slot + (ch << lpr_shift)] = make_uint4(L[2 * ch], M[2 * ch], L[2 * ch + 1], M[2 * ch + 1]);
    st.hib[slot + (ch << lpr_shift)] = make_uint2(H[2 * ch], H[2 * ch + 1]);
  }
}

// Stage code word w of token t from its kPer input values v (inactive
// threads pass zeros). The kGW = 64/kPer threads holding the words of one
// group must be kGW consecutive, aligned lanes of one warp, and all 32 lanes
// must call (the group maximum and the part sum are lane shuffles).
// lpr_shift = log2(LPR) (LPR is a power of two).
template <int BITS>
__device__ __forceinline__ void stage_word(const float (&v)[Geo<BITS>::kPer], bool active, int t, int w,
                                           const RowGeo& rg, int lpr_shift, const XStage& st) {
  using G = Geo<BITS>;
  constexpr int kGW = kGroup / G::kPer;
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < G::kPer; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
  for (int o = kGW / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  const int sh = x24_shift(m);
  const float sc = exp2i(sh);
  int X[G::kPer];
  int xsum = 0;
#pragma unroll
  for (int i = 0; i < G::kPer; ++i) {
    X[i] = x24_fix(v[i], sc);
    xsum += X[i];
  }
  if (active) store_word24<BITS>(X, t, w, rg, lpr_shift, st);
  // part sum over the 4 words of part p (4 consecutive lanes)
  xsum += __shfl_xor_sync(kFull, xsum, 1);
  xsum += __shfl_xor_sync(kFull, xsum, 2);
  if (active && (w & 3) == 0) {
    const float inv = exp2i(-sh);
    st.partinfo[t * rg.P + (w >> 2)] = make_float2(inv, (float)xsum * inv);
  }
}

// Stage T inputs of `cols` values into shared memory, one thread per code
// word: the 64/kPer consecutive threads of a group find the group maximum with
// shuffles, so a single pass with no block barrier inside does the job.
// All threads of the block must call; ends with __syncthreads().
template <int BITS, typename Src>
__device__ void stage_x24(const Src src, int T, int cols, XStage st) {
  using G = Geo<BITS>;
  const RowGeo rg = row_geo(cols, BITS);
  const int lpr_shift = __ffs(rg.LPR) - 1;
  const int words = cols * BITS / 32;
  const int total = T * words;  // a multiple of the group's words: groups never straddle a warp
  // t = floor(tw / words) through a float reciprocal: exact while total < 2^20
  // (the fraction of (tw + 0.5) / words stays >= 0.5 / words from an integer)
  const float inv_words = 1.f / (float)words;
  for (int base = 0; base < total; base += blockDim.x) {
    // uniform trip count per warp so that every shuffle sees all lanes
    const int tw = base + threadIdx.x;
    const bool active = tw < total;
    const int t = active ? (int)(((float)tw + 0.5f) * inv_words) : 0;
    const int w = active ? tw - t * words : 0;
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
    stage_word<BITS>(v, active, t, w, rg, lpr_shift, st);
  }
  __syncthreads();
}

// The same staging with two consecutive code words per thread: half the
// threads, so T * words <= 2 * blockDim.x takes a single pass. A group's words
// sit on kGW/2 consecutive lanes and a part's 4 words on 2, so the group
// maximum, the shifts and the part sums, hence every staged byte, equal
// stage_x24's. All threads of the block must call; ends with __syncthreads().
template <int BITS, typename Src>
__device__ __forceinline__ void stage_x24_pairs(const Src src, int T, int cols, XStage st) {
  using G = Geo<BITS>;
  constexpr int kGL = kGroup / G::kPer / 2;  // lanes per group
  const RowGeo rg = row_geo(cols, BITS);
  const int lpr_shift = __ffs(rg.LPR) - 1;
  const int hw = cols * BITS / 64;  // word pairs per input (cols is a multiple of 64)
  const int total = T * hw;
  const float inv_hw = 1.f / (float)hw;  // exact floor below, as in stage_x24
  for (int base = 0; base < total; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const bool active = i < total;
    const int t = active ? (int)(((float)i + 0.5f) * inv_hw) : 0;
    const int w0 = active ? 2 * (i - t * hw) : 0;
    float v[2 * G::kPer];
#pragma unroll
    for (int k = 0; k < 2 * G::kPer; k += 8) {
      if (active) {
        src.load8(t, w0 * G::kPer + k, v + k);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[k + j] = 0.f;
      }
    }
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 2 * G::kPer; ++k) m = fmaxf(m, fabsf(v[k]));
#pragma unroll
    for (int o = kGL / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    const int sh = x24_shift(m);
    const float sc = exp2i(sh);
    int xsum = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int X[G::kPer];
#pragma unroll
      for (int k = 0; k < G::kPer; ++k) {
        X[k] = x24_fix(v[h * G::kPer + k], sc);
        xsum += X[k];
      }
      if (active) store_word24<BITS>(X, t, w0 + h, rg, lpr_shift, st);
    }
    xsum += __shfl_xor_sync(kFull, xsum, 1);  // the part's other word pair
    if (active && (w0 & 3) == 0) {
      const float inv = exp2i(-sh);
      st.partinfo[t * rg.P + (w0 >> 2)] = make_float2(inv, (float)xsum * inv);
    }
  }
  __syncthreads();
}

// Integer dot product of one part (4 code words) with its staged input bytes
// (xc[c*NCH + ch]: L and M bytes, xh[...]: H bytes) and part info pi. Returns
// s*2^-sh*sum(q*X) + b*2^-sh*sum(X) added to acc.
template <int BITS>
__device__ __forceinline__ float part_dot_x(const uint4 qv, uint32_t sbw, const uint4 (&xc)[4 * Geo<BITS>::kNch],
                                            const uint2 (&xh)[4 * Geo<BITS>::kNch], const float2 pi, float acc) {
  using G = Geo<BITS>;
  const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
  int lo, hi;
  if (BITS == 4) {
    // odd codes stay in the high nibbles (16x their value) and get their own
    // accumulators, divided by 16 at the end (exact: every term is a multiple
    // of 16); saves the shift per word.
    uint32_t l0 = 0, l1 = 0, m0 = 0, m1 = 0;
    int h0 = 0, h1 = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 x = xc[c];
      const uint2 xhh = xh[c];
      const uint32_t v0 = qw[c] & 0x0f0f0f0fu, v1 = qw[c] & 0xf0f0f0f0u;
      l0 = dp4a_uu(v0, x.x, l0);
      m0 = dp4a_uu(v0, x.y, m0);
      h0 = dp4a_us(v0, xhh.x, h0);
      l1 = dp4a_uu(v1, x.z, l1);
      m1 = dp4a_uu(v1, x.w, m1);
      h1 = dp4a_us(v1, xhh.y, h1);
    }
    lo = (int)(l0 + (l1 >> 4)) + (int)(m0 + (m1 >> 4)) * 256;  // < 2^25
    hi = h0 + (h1 >> 4);
  } else {
    uint32_t l = 0, m = 0;
    int h = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int ch = 0; ch < G::kNch; ++ch) {
        const uint4 x = xc[c * G::kNch + ch];
        const uint2 xhh = xh[c * G::kNch + ch];
        const uint32_t v0 = (qw[c] >> (BITS * (2 * ch))) & G::kByteMask;
        const uint32_t v1 = (qw[c] >> (BITS * (2 * ch + 1))) & G::kByteMask;
        l = dp4a_uu(v0, x.x, l);
        m = dp4a_uu(v0, x.y, m);
        h = dp4a_us(v0, xhh.x, h);
        l = dp4a_uu(v1, x.z, l);
        m = dp4a_uu(v1, x.w, m);
        h = dp4a_us(v1, xhh.y, h);
      }
    }
    lo = (int)l + (int)m * 256;
    hi = h;
  }
  const float A = fmaf((float)hi, 65536.f, (float)lo);
  const float s = bf16lo(sbw), b = bf16hi(sbw);
  return fmaf(s * pi.x, A, fmaf(b, pi.y, acc));
}

// The staged input bytes of part p = it*LPR + lp of token t.
template <int BITS>
__device__ __forceinline__ void load_part_x(const XStage& st, int t, int it, int lp, const RowGeo& rg,
                                            uint4 (&xc)[4 * Geo<BITS>::kNch], uint2 (&xh)[4 * Geo<BITS>::kNch]) {
  const int base = ((t * rg.NIT + it) * 4 * Geo<BITS>::kNch) * rg.LPR + lp;
#pragma unroll
  for (int i = 0; i < 4 * Geo<BITS>::kNch; ++i) {
    xc[i] = st.chunks[base + i * rg.LPR];
    xh[i] = st.hib[base + i * rg.LPR];
  }
}

// Integer dot product of one part (4 code words) with staged token t.
// The part is p = it*LPR + lp (iteration it of lane lp of the row).
template <int BITS>
__device__ __forceinline__ float part_dot24(const uint4 qv, uint32_t sbw, const XStage& st, int t, int it, int lp,
                                            const RowGeo& rg, float acc) {
  uint4 xc[4 * Geo<BITS>::kNch];
  uint2 xh[4 * Geo<BITS>::kNch];
  load_part_x<BITS>(st, t, it, lp, rg, xc, xh);
  return part_dot_x<BITS>(qv, sbw, xc, xh, st.partinfo[t * rg.P + it * rg.LPR + lp], acc);
}

// Group index of part p.
template <int BITS>
__device__ __forceinline__ int part_group(int p) {
  return BITS == 4 ? (p >> 1) : p;
}

// Sum over the LPR lanes that share a row (lanes l, l^1, ... within the row's span).
__device__ __forceinline__ float row_reduce(float v, int LPR) {
  for (int o = LPR >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// row_reduce of four values at once (LPR >= 4), the same scheme as
// row_reduce8 below with two halving stages. Returns the sum of value
// u = 2*[lane & LPR/2] + [lane & LPR/4].
__device__ __forceinline__ float row_reduce4(float (&v)[4], int LPR, int lane) {
  int o = LPR >> 1;
  bool up = (lane & o) != 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = up ? v[j + 2] : v[j], send = up ? v[j] : v[j + 2];
    v[j] = keep + __shfl_xor_sync(kFull, send, o);
  }
  o >>= 1;
  up = (lane & o) != 0;
  {
    const float keep = up ? v[1] : v[0], send = up ? v[0] : v[1];
    v[0] = keep + __shfl_xor_sync(kFull, send, o);
  }
  for (o >>= 1; o > 0; o >>= 1) v[0] += __shfl_xor_sync(kFull, v[0], o);
  return v[0];
}

// row_reduce of eight values at once (LPR >= 8). Each of the first three
// stages halves the values a lane holds: the lane keeps one half, sends the
// other to its partner and adds the partner's copy of the half it kept. Every
// addition pairs the same two lanes' partial sums as row_reduce does, in the
// same order, so each result is bit-identical to row_reduce(v[u], LPR).
// Returns the sum of value u = 4*[lane & LPR/2] + 2*[lane & LPR/4] +
// [lane & LPR/8] (each bracket 0 or 1), held by every lane with those bits.
__device__ __forceinline__ float row_reduce8(float (&v)[8], int LPR, int lane) {
  int o = LPR >> 1;
  bool up = (lane & o) != 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = up ? v[j + 4] : v[j], send = up ? v[j] : v[j + 4];
    v[j] = keep + __shfl_xor_sync(kFull, send, o);
  }
  o >>= 1;
  up = (lane & o) != 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = up ? v[j + 2] : v[j], send = up ? v[j] : v[j + 2];
    v[j] = keep + __shfl_xor_sync(kFull, send, o);
  }
  o >>= 1;
  up = (lane & o) != 0;
  {
    const float keep = up ? v[1] : v[0], send = up ? v[0] : v[1];
    v[0] = keep + __shfl_xor_sync(kFull, send, o);
  }
  for (o >>= 1; o > 0; o >>= 1) v[0] += __shfl_xor_sync(kFull, v[0], o);
  return v[0];
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (sm_90+). A kernel launched with
// launch_overlapped() may start while the previous kernel on its stream is
// still running. Before pdl_wait() it reads only data that no earlier kernel
// writes (the weights); pdl_wait() blocks until every earlier kernel on the
// stream has completed and its writes are visible; inputs are read and outputs
// written after that. pdl_trigger() comes right after the wait, so the next
// kernel starts its prologue only once this one runs: at most one kernel waits
// on the SMs behind the running one (triggering at the start let a chain of
// waiting kernels fill the SMs and slowed the running one).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_overlapped(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace bgq
