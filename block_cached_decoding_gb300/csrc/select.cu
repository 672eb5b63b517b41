// Merge of the per-split vocabulary partials into confidence / log-odds /
// argmax, followed by the unmask decision for one block per sequence.
// One CTA per sequence.  Selection ranks masked positions by kappa =
// log((1 - c) / c) (lowest position first on ties):
//   threshold: kappa_i < kappa_tau (i.e. c_i > tau); none -> rank 0 only
//   factor:    largest n with (n + 1) (1 - c_(n)) < f, at least one
//   top-k:     ranks < k
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxBlock = 256;
constexpr int kMaxSplitsPerLane = 10;  // splits <= 320 handled with independent preloads

__global__ void __launch_bounds__(kThreads)
    select_kernel(SelectProblem p, const VocabStat *__restrict__ part, int splits) {
  __shared__ int mpos[kMaxBlock];
  __shared__ float kap[kMaxBlock];
  __shared__ float cf[kMaxBlock];
  __shared__ int tok[kMaxBlock];
  __shared__ int s_m, s_any, s_nbest, s_nsel;
  // launched as a programmatic dependent of the LM-head kernel: wait for its partials
  tc::pdl_wait_primary();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B;
  const int32_t *trow = p.tokens + (int64_t)b * p.seq_len + p.s;

  if (tid == 0) { s_any = 0; s_nbest = 0; s_nsel = 0; }
  // this sequence's masked positions in order
  if (warp == 0) {
    int base = 0;
    for (int c = 0; c < B; c += 32) {
      const int i = c + lane;
      const bool m = i < B && trow[i] == p.mask_id;
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (m) mpos[base + __popc(bal & ((1u << lane) - 1u))] = i;
      base += __popc(bal);
    }
    if (lane == 0) s_m = base;
  }
  for (int i = tid; i < B; i += kThreads) { kap[i] = __int_as_float(0x7fffffff); cf[i] = kap[i]; tok[i] = -1; }
  __syncthreads();
  const int M = s_m;

  // merge the splits of each masked row (partials indexed by block row b * B + i):
  // one warp per row, fixed reduction tree
  for (int j = warp; j < M; j += kThreads / 32) {
    const VocabStat *pr = part + ((int64_t)b * B + mpos[j]) * splits;
    VocabStat acc = vs_identity();
    if (splits <= 32 * kMaxSplitsPerLane) {
      // issue every load of this lane before merging, so their latencies overlap
      VocabStat v[kMaxSplitsPerLane];
#pragma unroll
      for (int k = 0; k < kMaxSplitsPerLane; ++k) {
        const int g = lane + 32 * k;
        v[k] = g < splits ? pr[g] : vs_identity();
      }
#pragma unroll
      for (int k = 0; k < kMaxSplitsPerLane; ++k) acc = vs_merge(acc, v[k]);
    } else {
      for (int g = lane; g < splits; g += 32) acc = vs_merge(acc, pr[g]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = vs_merge(acc, vs_shfl_xor(acc, o));
    if (lane == 0) {
      const int i = mpos[j];
      const float k = vs_kappa(acc);
      kap[i] = k;
      cf[i] = 1.f / (1.f + __expf(k));
      tok[i] = acc.a1;
    }
  }
  __syncthreads();

  // rank among masked positions by (kappa, position)
  bool masked = false, sel = false;
  int rank = 0;
  const int i = tid;
  if (i < B) {
    masked = tok[i] >= 0;
    if (masked) {
      const float ki = kap[i];
      for (int j = 0; j < M; ++j) {
        const int pj = mpos[j];
        const float kj = kap[pj];
        rank += (kj < ki) || (kj == ki && pj < i);
      }
    }
  }
  if (p.strategy == FDLLM_SELECT_THRESHOLD) {
    sel = masked && kap[i < B ? i : 0] < p.kappa_tau;
    if (sel) s_any = 1;
    __syncthreads();
    if (!s_any) sel = masked && rank == 0;
  } else if (p.strategy == FDLLM_SELECT_FACTOR) {
    if (masked) {
      const float eps = 1.f / (1.f + __expf(-kap[i]));  // 1 - c
      if ((float)(rank + 2) * eps < p.factor) atomicMax(&s_nbest, rank + 1);
    }
    __syncthreads();
    sel = masked && rank < max(s_nbest, 1);
  } else {
    sel = masked && rank < p.topk;
  }
  if (i < B) {
    const int64_t o = (int64_t)b * B + i;
    p.unmasked[o] = sel ? 1 : 0;
    p.conf[o] = masked ? cf[i] : __int_as_float(0x7fffffff);
    if (p.kappa) p.kappa[o] = masked ? kap[i] : __int_as_float(0x7fffffff);
    p.argmax[o] = masked ? tok[i] : -1;
    if (sel) {
      p.tokens[(int64_t)b * p.seq_len + p.s + i] = tok[i];
      atomicAdd(&s_nsel, 1);
    }
  }
  __syncthreads();
  if (tid == 0) p.n_left[b] = M - s_nsel;
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
