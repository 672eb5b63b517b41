// KV cache splice / refresh: cache[:, start : start + len] <- src for K and V.
// Pure data movement, bound by HBM bandwidth: 16-byte vector copies over a
// grid sized to the SM count, both tensors in one launch.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {

__global__ void __launch_bounds__(256) splice_kernel(int batch, int64_t cache_vecs_per_b,
                                                      int64_t start_vec, int64_t len_vecs,
                                                      uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                                      const uint4 *__restrict__ ks,
                                                      const uint4 *__restrict__ vs,
                                                      const int32_t *__restrict__ starts, int64_t row_vecs,
                                                      int max_start, int32_t *err) {
  // launched as a programmatic dependent: the sources may come from the previous kernel in the
  // stream, which may also still read the cache rows written here
  tc::pdl_wait_primary();
  tc::pdl_launch_dependents();
  const int64_t per_tensor = (int64_t)batch * len_vecs;
  const int64_t total = 2 * per_tensor;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= per_tensor;
    const int64_t j = is_v ? i - per_tensor : i;
    const int64_t b = j / len_vecs;
    const int64_t r = j - b * len_vecs;
    int64_t sv = start_vec;
    if (starts != nullptr) {                       // sequence b's own window
      const int sb = starts[b];
      if (sb < 0 || sb > max_start) {
        if (r == 0 && !is_v) record_device_error(err, 233);
        continue;
      }
      sv = (int64_t)sb * row_vecs;
    }
    const uint4 x = __ldcs((is_v ? vs : ks) + j);  // streamed once
    uint4 *dst = (is_v ? vc : kc) + b * cache_vecs_per_b + sv + r;
    *dst = x;
  }
}

cudaError_t launch_splice(int batch, int64_t cache_rows, int64_t row_bytes, int64_t start,
                          int64_t len, void *kc, void *vc, const void *ks, const void *vs,
                          cudaStream_t st, const int32_t *starts, int32_t *err) {
  const int64_t rv = row_bytes / 16;
  const int64_t total = 2 * (int64_t)batch * len * rv;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, splice_kernel, batch, cache_rows * rv, start * rv, len * rv,
                                           (uint4 *)kc, (uint4 *)vc, (const uint4 *)ks, (const uint4 *)vs,
                                           starts, rv, (int)(cache_rows - len), err);
  count_launches(1);
  return e;
}

}  // namespace fdllm
