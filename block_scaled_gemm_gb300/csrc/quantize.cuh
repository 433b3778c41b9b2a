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
template <typename T>
__global__ void mx_quantize_rows_kernel(const T *__restrict__ X, int64_t nblocks,
                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;  // lane within the block's four
  const int64_t groups = (nblocks + 7) / 8;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       gw < groups; gw += warps) {
    const int64_t b = gw * 8 + (lane >> 2);
    const bool live = b < nblocks;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    if (live) {
      const T *src = X + b * 32 + sub * 8;
      if constexpr (sizeof(T) == 4) {
        const float4 q0 = reinterpret_cast<const float4 *>(src)[0];
        const float4 q1 = reinterpret_cast<const float4 *>(src)[1];
        v[0] = q0.x; v[1] = q0.y; v[2] = q0.z; v[3] = q0.w;
        v[4] = q1.x; v[5] = q1.y; v[6] = q1.z; v[7] = q1.w;
      } else {
        const uint4 q = *reinterpret_cast<const uint4 *>(src);
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
    uint32_t w0 = mx_e4m3x2(v[0] * m, v[1] * m) | (mx_e4m3x2(v[2] * m, v[3] * m) << 16);
    uint32_t w1 = mx_e4m3x2(v[4] * m, v[5] * m) | (mx_e4m3x2(v[6] * m, v[7] * m) << 16);
    if (live) {
      *reinterpret_cast<uint2 *>(codes + b * 32 + sub * 8) = make_uint2(w0, w1);
      if (sub == 0) scales[b] = static_cast<uint8_t>(s);
    }
  }
}

// Blocks down the columns (X is R x C, R % 32 == 0; scales C x R/32, row j
// for column j): one thread per (NC adjacent columns, 32-row block);
// neighbouring threads take neighbouring column pairs, so every row access
// of a warp is contiguous, NC x 32 x sizeof(T) bytes wide.  The thread holds
// its 32 rows as loaded words (all loads issued before the first use) and
// stores NC codes per row.  NC = 2 needs C even.
template <typename T, int NC>
__global__ void mx_quantize_cols_kernel(const T *__restrict__ X, int64_t R, int64_t C,
                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
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
    Word raw[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) raw[e] = *reinterpret_cast<const Word *>(src + e * C);
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
      if constexpr (NC == 2)
        *reinterpret_cast<uint16_t *>(dst + e * C) = static_cast<uint16_t>(
            mx_e4m3x2(mx_to_float<T>(t[0]) * m[0], mx_to_float<T>(t[1]) * m[1]));
      else
        dst[e * C] = static_cast<uint8_t>(mx_e4m3(mx_to_float<T>(t[0]) * m[0]));
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) scales[(j + c) * rblocks + rb] = static_cast<uint8_t>(s[c]);
  }
}

}  // namespace mxg
