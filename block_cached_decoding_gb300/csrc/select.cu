// Standalone merge + select kernel (one CTA per sequence), used after the
// CUDA-core LM head; the tensor-core LM head runs the same per-sequence code
// in its own tail (select_impl.cuh).
#include "common.cuh"
#include "internal.h"
#include "select_impl.cuh"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads)
    select_kernel(SelectProblem p, const VocabStat *__restrict__ part, int splits) {
  __shared__ SelectScratch sc;
  // launched as a programmatic dependent of the LM-head kernel: wait for its partials
  tc::pdl_wait_primary();
  select_sequence<kThreads>(p, part, splits, blockIdx.x, sc);
}

}  // namespace

cudaError_t launch_select(const SelectProblem &p, const VocabStat *part, int splits, cudaStream_t st) {
  // programmatic dependent launch: the CTAs become resident while the LM-head
  // kernel drains and wait for its memory inside the kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, select_kernel, p, part, splits);
  count_launches(1);
  return e;
}

}  // namespace fdllm
