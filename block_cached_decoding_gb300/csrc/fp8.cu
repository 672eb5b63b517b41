// Per-row E4M3 quantisation for the FP8 weight cache, the block's hidden rows and the FP8 KV cache:
// the rule of fp8_rule.cuh, one CTA per row (grid-stride over rows); a pure streaming kernel.
#include <cuda_fp8.h>

#include "common.cuh"
#include "fp8_rule.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 256;

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
  __shared__ float red[kThreads / 32];
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
    fp8rule::quantize_row<kThreads>(src + (bb * src_bstride + rr) * cols, cols, q + r * cols, scale + r, vec, red);
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
