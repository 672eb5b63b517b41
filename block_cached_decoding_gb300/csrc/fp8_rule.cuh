// The per-row E4M3 quantisation rule, shared by the row quantiser kernel and the FP8-weight LM head
// (which quantises the block's hidden rows itself).  Row r gets the scale 2^k, k the smallest integer
// with max|row| <= 448 * 2^k (448 is E4M3's largest finite value; k = 0 for an all-zero row), and the
// codes round(x / 2^k) to the nearest E4M3 value, ties to even.  The division is an exact exponent
// shift, and k is decided exactly from the binary exponent of max|row| (max|row| = f 2^x, f in
// [0.5, 1); 448 = 0.875 * 2^9), so the codes do not depend on how the maximum or the shift is
// evaluated.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace fdllm {
namespace fp8rule {

// x * 2^-k exactly for the k of this rule (|k| <= 252): two power-of-two factors, each a normal
// float, so neither product rounds (the result is at most 448 in magnitude; a product below the
// normal range only arises for values that round to a zero code either way)
struct Shift {
  float f1, f2;
  __device__ explicit Shift(int k) {
    const int a = -k / 2, b = -k - a;                  // 2^a * 2^b = 2^-k, |a|, |b| <= 126
    f1 = __int_as_float((127 + a) << 23);
    f2 = __int_as_float((127 + b) << 23);
  }
  __device__ float operator()(float x) const { return __fmul_rn(__fmul_rn(x, f1), f2); }
};

__device__ __forceinline__ int scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int x;
  const float f = frexpf(amax, &x);
  return f <= 0.875f ? x - 9 : x - 8;
}

__device__ __forceinline__ uint16_t cvt2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// 16-byte vectors of the source: 8 bf16 or 4 fp32
__device__ __forceinline__ void unpack(const uint4 &u, float (&x)[8], const __nv_bfloat16 *) {
  const __nv_bfloat162 *h = (const __nv_bfloat162 *)&u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void unpack(const uint4 &u, float (&x)[8], const float *) {
  x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y); x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
}

// One row of `cols` values quantised by all NT threads of the CTA: codes into qrow, 2^k into *scale.
// `vec`: the row and its codes start on 16-byte boundaries and cols % 16 == 0 (16-byte vectors).
// red: NT / 32 floats of shared memory; the call ends with a barrier, so red may be reused after it.
template <int NT, typename T>
__device__ __forceinline__ void quantize_row(const T *__restrict__ row, int cols, uint8_t *__restrict__ qrow,
                                             float *scale, bool vec, float *red) {
  constexpr int VE = 16 / (int)sizeof(T);               // elements per 16-byte vector
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = 0.f;
  if (vec) {
    for (int i = threadIdx.x * VE; i < cols; i += NT * VE) {
      float x[8];
      unpack(*(const uint4 *)(row + i), x, row);
#pragma unroll
      for (int e = 0; e < VE; ++e) m = fmaxf(m, fabsf(x[e]));
    }
  } else {
    for (int i = threadIdx.x; i < cols; i += NT) m = fmaxf(m, fabsf(to_f32(row[i])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) amax = fmaxf(amax, red[w]);
  const int k = scale_exponent(amax);
  const Shift sh(k);
  if (threadIdx.x == 0) *scale = ldexpf(1.f, k);
  if (vec) {
    for (int i = threadIdx.x * VE; i < cols; i += NT * VE) {
      float x[8];
      unpack(*(const uint4 *)(row + i), x, row);
      if constexpr (VE == 8) {
        uint4 o;
        o.x = cvt2(sh(x[0]), sh(x[1])) | ((uint32_t)cvt2(sh(x[2]), sh(x[3])) << 16);
        o.y = cvt2(sh(x[4]), sh(x[5])) | ((uint32_t)cvt2(sh(x[6]), sh(x[7])) << 16);
        *(uint2 *)(qrow + i) = make_uint2(o.x, o.y);
      } else {
        *(uint32_t *)(qrow + i) = cvt2(sh(x[0]), sh(x[1])) | ((uint32_t)cvt2(sh(x[2]), sh(x[3])) << 16);
      }
    }
  } else {
    for (int i = threadIdx.x; i < cols; i += NT)
      qrow[i] = (uint8_t)__nv_cvt_float_to_fp8(sh(to_f32(row[i])), __NV_SATFINITE, __NV_E4M3);
  }
  __syncthreads();   // red may be rewritten after this
}

}  // namespace fp8rule
}  // namespace fdllm
