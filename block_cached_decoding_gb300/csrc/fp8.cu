// Per-row E4M3 quantisation for the FP8 weight cache.
//
// Row r of a bf16 / fp32 matrix gets the scale 2^k with k the smallest integer such
// that max|row| <= 448 * 2^k (448 is E4M3's largest finite value; k = 0 for an
// all-zero row) and the codes round(x / 2^k) to the nearest E4M3 value, ties to
// even.  The division is an exact exponent shift, and k is decided exactly from
// the binary exponent of max|row| (max|row| = f 2^x, f in [0.5, 1); 448 = 0.875 * 2^9),
// so the codes do not depend on how the maximum or the shift is evaluated.  One CTA
// per row (grid-stride over rows); a pure streaming kernel.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 256;

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

// Rows R = bb * rpb + r (bb < batch): source row bb * src_bstride + r, destination row (codes and
// scale) bb * dst_bstride + r, plus starts[bb] * row_step when a per-sequence start array is given (a
// start outside [0, max_start] skips the sequence and records device error 233).
template <typename T>
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const T *__restrict__ src, int64_t rows, int cols,
                                                                 uint8_t *__restrict__ q, float *__restrict__ scale,
                                                                 int64_t rpb, int64_t src_bstride,
                                                                 int64_t dst_bstride, const int32_t *starts,
                                                                 int64_t row_step, int max_start, int32_t *err) {
  // launched as a programmatic dependent: the source may come from the previous kernel in the stream
  tc::pdl_wait_primary();
  tc::pdl_launch_dependents();
  constexpr int VE = 16 / (int)sizeof(T);               // elements per 16-byte vector
  __shared__ float red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // whole 16-byte vectors when every row starts on a 16-byte boundary (and its codes on VE bytes)
  const bool vec = cols % 16 == 0 && ((uintptr_t)src & 15) == 0 && ((uintptr_t)q & 15) == 0;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t bb = R / rpb, rr = R - bb * rpb;
    int64_t r = bb * dst_bstride + rr;                 // destination row
    if (starts != nullptr) {                           // uniform across the CTA: one row per CTA
      const int sb = starts[bb];
      if (sb < 0 || sb > max_start) {
        if (threadIdx.x == 0 && rr == 0) record_device_error(err, 233);
        continue;
      }
      r += (int64_t)sb * row_step;
    }
    const T *row = src + (bb * src_bstride + rr) * cols;
    uint8_t *qrow = q + r * cols;
    float m = 0.f;
    if (vec) {
      for (int i = threadIdx.x * VE; i < cols; i += kThreads * VE) {
        float x[8];
        unpack(*(const uint4 *)(row + i), x, row);
#pragma unroll
        for (int e = 0; e < VE; ++e) m = fmaxf(m, fabsf(x[e]));
      }
    } else {
      for (int i = threadIdx.x; i < cols; i += kThreads) m = fmaxf(m, fabsf(to_f32(row[i])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float amax = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const int k = scale_exponent(amax);
    const Shift sh(k);
    if (threadIdx.x == 0) scale[r] = ldexpf(1.f, k);
    if (vec) {
      for (int i = threadIdx.x * VE; i < cols; i += kThreads * VE) {
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
      for (int i = threadIdx.x; i < cols; i += kThreads)
        qrow[i] = (uint8_t)__nv_cvt_float_to_fp8(sh(to_f32(row[i])), __NV_SATFINITE, __NV_E4M3);
    }
    __syncthreads();   // red is rewritten for the next row
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void *src, bool src_bf16, int64_t rows, int cols, uint8_t *q, float *scale,
                                cudaStream_t st) {
  return launch_quantize_fp8_batched(src, src_bf16, 1, rows, cols, rows, q, scale, rows, st, nullptr, 0, 0, nullptr);
}

cudaError_t launch_quantize_fp8_batched(const void *src, bool src_bf16, int64_t batch, int64_t rpb, int cols,
                                        int64_t src_bstride, uint8_t *q, float *scale, int64_t dst_bstride,
                                        cudaStream_t st, const int32_t *starts, int64_t row_step, int max_start,
                                        int32_t *err) {
  const int64_t rows = batch * rpb;
  if (rows == 0 || cols == 0) return cudaSuccess;
  int64_t grid = rows;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (src_bf16)
    e = cudaLaunchKernelEx(&cfg, quantize_rows_kernel<__nv_bfloat16>, (const __nv_bfloat16 *)src, rows, cols, q,
                           scale, rpb, src_bstride, dst_bstride, starts, row_step, max_start, err);
  else
    e = cudaLaunchKernelEx(&cfg, quantize_rows_kernel<float>, (const float *)src, rows, cols, q, scale, rpb,
                           src_bstride, dst_bstride, starts, row_step, max_start, err);
  count_launches(1);
  return e;
}

}  // namespace fdllm
