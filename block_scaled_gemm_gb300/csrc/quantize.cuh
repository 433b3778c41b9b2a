// quantize.cuh -- MX quantization on the GPU: a real matrix (FP32 or BF16)
// to E4M3 codes with one E8M0 scale per 32 values, the form the GEMM takes.
//
// Per block of 32 values (OCP Microscaling Formats v1.0 conversion, E4M3
// maximum 448):
//   scale  = clamp(127 + ceil(log2(amax / 448)), 0, 254), 127 when amax = 0
//   code_i = E4M3(clamp(x_i * 2^(127 - scale), -448, 448)), round to nearest
//            even, sign kept
// The scaling multiplies by a power of two in FP32, exact wherever the
// result can round to a nonzero code; the E4M3 rounding is the hardware
// conversion (round to nearest even, saturating at +-448, which equals the
// clamp).  Inputs must be finite.
//
// Stochastic rounding (the FP32 -> FP8 rounding with caller-supplied random
// bits of "TLX API Quick Reference", section "Utility", `tlx.stoch_round`):
// each value has its own 32-bit random word r, and the scaled FP32 value
// y = x * 2^(127 - scale) rounds to the E4M3 magnitude above |y| with
// probability (|y| - lo) / q, lo the E4M3 magnitude below and q the spacing
// there, decided exactly as r < 2^32 (|y| - lo) / q (see mx_e4m3_sr).
//
// HBM-bound: each value is read once and its code written once.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace mxg {

// smallest integer t with amax <= 448 * 2^t (amax > 0), exact:
// amax = f * 2^E with f in [0.5, 1) and 448 * 2^t = 0.875 * 2^(t + 9)
__device__ __forceinline__ int mx_scale_of(float amax) {
  if (!(amax > 0.0f)) return 127;
  int E;
  const float f = frexpf(amax, &E);
  const int t = f <= 0.875f ? E - 9 : E - 8;
  return min(max(127 + t, 0), 254);
}

// 2^(127 - s) as an FP32 multiplier.  For finite FP32 or BF16 inputs
// amax <= FLT_MAX gives s <= 127 + 120 = 247, so 2^(127 - s) >= 2^-120 is a
// normal number; s = 254 would need amax > 448 * 2^126.
__device__ __forceinline__ float mx_pow2(int s) { return __int_as_float((254 - s) << 23); }

// E4M3 codes of two values, rounded to nearest even and saturated to +-448
// (the same as clamping first, 448 being representable); byte 0 holds a.
__device__ __forceinline__ uint32_t mx_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ uint32_t mx_e4m3(float y) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
}

// E4M3 code of y by stochastic rounding with the random word r.  |y| is
// clamped to 448 and written m * 2^-sh * q with q = 2^qe the E4M3 spacing at
// |y| (2^(e-3) in the binade [2^e, 2^(e+1)) for e >= -6, else 2^-9) and m the
// FP32 significand; lo = floor(m / 2^sh) q, and the rounding goes up when
// r * 2^sh < rem * 2^32, rem = m mod 2^sh.  32-bit integer arithmetic, exact.
//   |y| >= 2^-6 (E4M3 normal): sh = 20, so lo is |y| with the low 20 FP32
//   mantissa bits cleared, the test is r < rem * 2^12, and rounding up adds
//   one unit of the 21st bit (a carry into the exponent is the next binade).
//   The FP32 encoding of the result then maps to the E4M3 code directly:
//   exponent - 120 and the top three mantissa bits.
//   |y| < 2^-6 (subnormal grid, q = 2^-9): sh = 21..140; for sh <= 32 the
//   test is r < rem * 2^(32-sh) (below 2^32, as rem < 2^sh), for sh = 32 + t
//   it is r < ceil(rem / 2^t), which is 1 once 2^t > rem.
// The sign is kept, also for zero.
__device__ __forceinline__ uint32_t mx_e4m3_sr(float y, uint32_t r) {
  const uint32_t bits = __float_as_uint(y);
  const uint32_t sign = (bits >> 24) & 0x80u;
  const uint32_t a = min(bits & 0x7FFFFFFFu, 0x43E00000u);  // 0x43E00000 = 448.0f
  if (a >= 0x3C800000u) {                                    // 0x3C800000 = 2^-6
    const uint32_t v = (a & ~0xFFFFFu) + (r < ((a & 0xFFFFFu) << 12) ? 0x100000u : 0u);
    return sign | ((v >> 20) - (120u << 3));
  }
  const int be = static_cast<int>(a >> 23);                 // 0 when FP32-subnormal
  const uint32_t m = be ? (a & 0x7FFFFFu) | 0x800000u : a;  // |y| = m * 2^(max(be,1) - 150)
  const int sh = 141 - max(be, 1);                          // log2(2^-9 / 2^(max(be,1) - 150))
  const uint32_t n = sh < 32 ? m >> sh : 0u;                // |y| / 2^-9, rounded down (< 8)
  const uint32_t rem = sh < 32 ? m & ((1u << sh) - 1u) : m;
  bool up;
  if (sh <= 32) {
    up = r < (rem << (32 - sh));
  } else {
    const int t = sh - 32;  // rem = m < 2^24
    up = t < 24 ? r < ((rem + (1u << t) - 1u) >> t) : (r == 0u && rem != 0u);
  }
  return sign | (n + (up ? 1u : 0u));  // 8 is the code of 2^-6 too
}

// Packed scale layout (the order the GEMM's tensor cores read): byte of the
// scale of row r (A, blocks along rows) or column c (B, blocks down
// columns) for K block kb, with S K steps of 128.  A: chunk (r / 128, kb / 4)
// at (r / 128 * S + kb / 4) * 512; B: chunk (c / 128, kb / 4) at
// ((c / 256 * S + kb / 4) * 2 + c / 128 % 2) * 512; inside a chunk, byte
// (r % 32) * 16 + (r / 32 % 4) * 4 + kb % 4.
__device__ __forceinline__ int64_t packed_row_scale_at(int64_t r, int64_t kb, int64_t S) {
  return ((r >> 7) * S + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}
__device__ __forceinline__ int64_t packed_col_scale_at(int64_t c, int64_t kb, int64_t S) {
  return (((c >> 8) * S + (kb >> 2)) * 2 + ((c >> 7) & 1)) * 512 + (c & 31) * 16 +
         ((c >> 5) & 3) * 4 + (kb & 3);
}

template <typename T>
__device__ __forceinline__ float mx_to_float(T v);
template <>
__device__ __forceinline__ float mx_to_float<float>(float v) { return v; }
template <>
__device__ __forceinline__ float mx_to_float<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// Blocks along the rows (X is R x C, C % 32 == 0; scales R x C/32): the
// blocks are contiguous in memory, block b = elements [32b, 32b + 32).
// Four lanes share a block, eight values each; a warp covers eight blocks.
// SR: rbits holds one random word per element, at the element's index.
// S > 0: the scales go to the packed layout with S K steps (a row has kbn
// blocks); S = 0: row-major, scale b for block b.
template <typename T, bool SR>
__global__ void mx_quantize_rows_kernel(const T *__restrict__ X, int64_t nblocks,
                                        const uint32_t *__restrict__ rbits,
                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                                        int64_t kbn, int64_t S) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;  // lane within the block's four
  const int64_t groups = (nblocks + 7) / 8;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       gw < groups; gw += warps) {
    const int64_t b = gw * 8 + (lane >> 2);
    const bool live = b < nblocks;
    float v[8];
    uint32_t r[8];  // random words (stochastic rounding), loaded with the values
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = 0.0f;
      r[e] = 0u;
    }
    if (live) {
      if constexpr (SR) {
        const uint4 r0 = reinterpret_cast<const uint4 *>(rbits + b * 32 + sub * 8)[0];
        const uint4 r1 = reinterpret_cast<const uint4 *>(rbits + b * 32 + sub * 8)[1];
        r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
        r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
      }
      // X is read once: evict-first loads (measured 2-5 % faster than
      // default-cached ones, BF16 more than FP32)
      const T *src = X + b * 32 + sub * 8;
      if constexpr (sizeof(T) == 4) {
        const float4 q0 = __ldcs(reinterpret_cast<const float4 *>(src));
        const float4 q1 = __ldcs(reinterpret_cast<const float4 *>(src) + 1);
        v[0] = q0.x; v[1] = q0.y; v[2] = q0.z; v[3] = q0.w;
        v[4] = q1.x; v[5] = q1.y; v[6] = q1.z; v[7] = q1.w;
      } else {
        const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(src));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = __uint_as_float(w[e] << 16);
          v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const int s = mx_scale_of(amax);
    const float m = mx_pow2(s);
    uint32_t w0, w1;
    if constexpr (SR) {
      uint32_t c[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = mx_e4m3_sr(v[e] * m, r[e]);
      w0 = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      w1 = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
    } else {
      w0 = mx_e4m3x2(v[0] * m, v[1] * m) | (mx_e4m3x2(v[2] * m, v[3] * m) << 16);
      w1 = mx_e4m3x2(v[4] * m, v[5] * m) | (mx_e4m3x2(v[6] * m, v[7] * m) << 16);
    }
    if (live) {
      *reinterpret_cast<uint2 *>(codes + b * 32 + sub * 8) = make_uint2(w0, w1);
      if (sub == 0) {
        const int64_t at = S ? packed_row_scale_at(b / kbn, b % kbn, S) : b;
        scales[at] = static_cast<uint8_t>(s);
      }
    }
  }
}

// Blocks down the columns (X is R x C, R % 32 == 0; scales C x R/32, row j
// for column j): one thread per (NC adjacent columns, 32-row block);
// neighbouring threads take neighbouring column pairs, so every row access
// of a warp is contiguous, NC x 32 x sizeof(T) bytes wide.  The thread holds
// its 32 rows as loaded words (all loads issued before the first use) and
// stores NC codes per row.  NC = 2 needs C even.  SR (NC = 1): rbits holds
// one random word per element, at the element's index; they are loaded with
// the values.
// S > 0: the scales go to the packed layout with S K steps; S = 0:
// C x R/32, row j for column j.
template <typename T, int NC, bool SR>
__global__ void mx_quantize_cols_kernel(const T *__restrict__ X, int64_t R, int64_t C,
                                        const uint32_t *__restrict__ rbits,
                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                                        int64_t S) {
  static_assert(NC == 1 || NC == 2, "one or two columns per thread");
  constexpr int kWordBytes = NC * static_cast<int>(sizeof(T));
  using Word = typename std::conditional<
      kWordBytes == 8, uint2,
      typename std::conditional<kWordBytes == 4, uint32_t, uint16_t>::type>::type;
  static_assert(sizeof(Word) == kWordBytes, "one load per row");
  const int64_t rblocks = R / 32;
  const int64_t groups = C / NC;
  const int64_t total = rblocks * groups;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t rb = i / groups, j = (i - rb * groups) * NC;
    const T *src = X + rb * 32 * C + j;
    static_assert(!SR || NC == 1, "stochastic rounding takes one column per thread");
    Word raw[32];
    uint32_t rw[SR ? 32 : 1];  // random words (stochastic rounding), loaded with the values
    const uint32_t *rsrc = SR ? rbits + rb * 32 * C + j : nullptr;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      raw[e] = *reinterpret_cast<const Word *>(src + e * C);
      if constexpr (SR) rw[e] = rsrc[e * C];
    }
    float amax[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) amax[c] = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const T *t = reinterpret_cast<const T *>(&raw[e]);
#pragma unroll
      for (int c = 0; c < NC; ++c) amax[c] = fmaxf(amax[c], fabsf(mx_to_float<T>(t[c])));
    }
    int s[NC];
    float m[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      s[c] = mx_scale_of(amax[c]);
      m[c] = mx_pow2(s[c]);
    }
    uint8_t *dst = codes + rb * 32 * C + j;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const T *t = reinterpret_cast<const T *>(&raw[e]);
      if constexpr (SR) {
        dst[e * C] = static_cast<uint8_t>(mx_e4m3_sr(mx_to_float<T>(t[0]) * m[0], rw[e]));
      } else if constexpr (NC == 2) {
        *reinterpret_cast<uint16_t *>(dst + e * C) = static_cast<uint16_t>(
            mx_e4m3x2(mx_to_float<T>(t[0]) * m[0], mx_to_float<T>(t[1]) * m[1]));
      } else {
        dst[e * C] = static_cast<uint8_t>(mx_e4m3(mx_to_float<T>(t[0]) * m[0]));
      }
    }
#pragma unroll
    for (int c = 0; c < NC; ++c)
      scales[S ? packed_col_scale_at(j + c, rb, S) : (j + c) * rblocks + rb] = static_cast<uint8_t>(s[c]);
  }
}

}  // namespace mxg
