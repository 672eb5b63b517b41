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

template <typename T>
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const T *__restrict__ src, int64_t rows, int cols,
                                                                 uint8_t *__restrict__ q, float *__restrict__ scale) {
  // launched as a programmatic dependent: the source may come from the previous kernel in the stream
  tc::pdl_wait_primary();
  tc::pdl_launch_dependents();
  __shared__ float red[kThreads / 32];
  __shared__ int kshift;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T *row = src + r * cols;
    float m = 0.f;
    for (int i = threadIdx.x; i < cols; i += kThreads) m = fmaxf(m, fabsf(to_f32(row[i])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float amax = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
      int k = 0;
      if (amax > 0.f) {
        int x;
        const float f = frexpf(amax, &x);
        k = f <= 0.875f ? x - 9 : x - 8;
      }
      kshift = k;
      scale[r] = ldexpf(1.f, k);
    }
    __syncthreads();
    const int k = kshift;
    uint8_t *qrow = q + r * cols;
    for (int i = threadIdx.x; i < cols; i += kThreads)
      qrow[i] = (uint8_t)__nv_cvt_float_to_fp8(ldexpf(to_f32(row[i]), -k), __NV_SATFINITE, __NV_E4M3);
    __syncthreads();   // red / kshift are rewritten for the next row
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void *src, bool src_bf16, int64_t rows, int cols, uint8_t *q, float *scale,
                                cudaStream_t st) {
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
                           scale);
  else
    e = cudaLaunchKernelEx(&cfg, quantize_rows_kernel<float>, (const float *)src, rows, cols, q, scale);
  count_launches(1);
  return e;
}

}  // namespace fdllm
