// Merge of the per-split vocabulary partials of one sequence's masked rows into
// confidence / log-odds / argmax, then the unmask decision for its block.
// Shared by select_kernel (one CTA per sequence) and the tail of the
// tensor-core LM-head kernel (the last CTAs to finish take one sequence each).
//
// Selection ranks masked positions by kappa = log((1 - c) / c), lowest
// position first on ties:
//   threshold: kappa_i < kappa_tau (i.e. c_i > tau); none -> rank 0 only
//   factor:    largest n with (n + 1) (1 - c_(n)) < f, at least one
//   top-k:     ranks < k
#pragma once

#include "common.cuh"
#include "internal.h"

namespace fdllm {

constexpr int kSelectMaxBlock = 256;
constexpr int kSelectMaxSplitsPerLane = 10;  // splits <= 320 merged with independent preloads

// A masked row's merged statistics (written by the LM-head tail, one warp per row).
struct RowStat {
  float kappa;
  int32_t token;
};

// Merge the `splits` partials of one row (called by a whole warp; lane 0 gets the result).
__device__ __forceinline__ VocabStat merge_row(const VocabStat *__restrict__ pr, int splits) {
  const int lane = threadIdx.x & 31;
  VocabStat acc = vs_identity();
  if (splits <= 32 * kSelectMaxSplitsPerLane) {
    VocabStat v[kSelectMaxSplitsPerLane];  // every load of this lane in flight before merging
#pragma unroll
    for (int k = 0; k < kSelectMaxSplitsPerLane; ++k) {
      const int g = lane + 32 * k;
      v[k] = g < splits ? pr[g] : vs_identity();
    }
#pragma unroll
    for (int k = 0; k < kSelectMaxSplitsPerLane; ++k) acc = vs_merge(acc, v[k]);
  } else {
    for (int g = lane; g < splits; g += 32) acc = vs_merge(acc, pr[g]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = vs_merge(acc, vs_shfl_xor(acc, o));
  return acc;
}

struct SelectScratch {
  int mpos[kSelectMaxBlock];
  float kap[kSelectMaxBlock];
  float cf[kSelectMaxBlock];
  int tok[kSelectMaxBlock];
  int m, any, nbest, nsel;
};

// Called by all NT threads of the CTA (NT >= block size, a multiple of 32).
// Either `part` holds the VocabStat partials [b * B + i][splits] and the rows are
// merged here, or `merged` (not null) already holds each masked row's RowStat.
template <int NT>
__device__ __forceinline__ void select_sequence(const SelectProblem &p, const VocabStat *__restrict__ part,
                                                int splits, int b, SelectScratch &sc,
                                                const RowStat *__restrict__ merged = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B;
  const int32_t *trow = p.tokens + (int64_t)b * p.seq_len + p.s;
  if (tid == 0) { sc.any = 0; sc.nbest = 0; sc.nsel = 0; }
  // this sequence's masked positions in order
  if (warp == 0) {
    int base = 0;
    for (int c = 0; c < B; c += 32) {
      const int i = c + lane;
      const bool m = i < B && trow[i] == p.mask_id;
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (m) sc.mpos[base + __popc(bal & ((1u << lane) - 1u))] = i;
      base += __popc(bal);
    }
    if (lane == 0) sc.m = base;
  }
  for (int i = tid; i < B; i += NT) {
    sc.kap[i] = __int_as_float(0x7fffffff);
    sc.cf[i] = sc.kap[i];
    sc.tok[i] = -1;
  }
  __syncthreads();
  const int M = sc.m;

  if (merged != nullptr) {
    for (int j = tid; j < M; j += NT) {
      const int i = sc.mpos[j];
      const RowStat rs = merged[(int64_t)b * B + i];
      sc.kap[i] = rs.kappa;
      sc.cf[i] = 1.f / (1.f + __expf(rs.kappa));
      sc.tok[i] = rs.token;
    }
  } else {
    // merge the splits of each masked row: one warp per row, fixed reduction tree
    for (int j = warp; j < M; j += NT / 32) {
      const VocabStat acc = merge_row(part + ((int64_t)b * B + sc.mpos[j]) * splits, splits);
      if (lane == 0) {
        const int i = sc.mpos[j];
        const float k = vs_kappa(acc);
        sc.kap[i] = k;
        sc.cf[i] = 1.f / (1.f + __expf(k));
        sc.tok[i] = acc.a1;
      }
    }
  }
  __syncthreads();

  // rank among masked positions by (kappa, position)
  bool masked = false, sel = false;
  int rank = 0;
  const int i = tid;
  if (i < B) {
    masked = sc.tok[i] >= 0;
    if (masked) {
      const float ki = sc.kap[i];
      for (int j = 0; j < M; ++j) {
        const int pj = sc.mpos[j];
        const float kj = sc.kap[pj];
        rank += (kj < ki) || (kj == ki && pj < i);
      }
    }
  }
  if (p.strategy == FDLLM_SELECT_THRESHOLD) {
    sel = masked && sc.kap[i < B ? i : 0] < p.kappa_tau;
    if (sel) sc.any = 1;
    __syncthreads();
    if (!sc.any) sel = masked && rank == 0;
  } else if (p.strategy == FDLLM_SELECT_FACTOR) {
    if (masked) {
      const float eps = 1.f / (1.f + __expf(-sc.kap[i]));  // 1 - c
      if ((float)(rank + 2) * eps < p.factor) atomicMax(&sc.nbest, rank + 1);
    }
    __syncthreads();
    sel = masked && rank < max(sc.nbest, 1);
  } else {
    sel = masked && rank < p.topk;
  }
  if (i < B) {
    const int64_t o = (int64_t)b * B + i;
    p.unmasked[o] = sel ? 1 : 0;
    p.conf[o] = masked ? sc.cf[i] : __int_as_float(0x7fffffff);
    if (p.kappa) p.kappa[o] = masked ? sc.kap[i] : __int_as_float(0x7fffffff);
    p.argmax[o] = masked ? sc.tok[i] : -1;
    if (sel) {
      p.tokens[(int64_t)b * p.seq_len + p.s + i] = sc.tok[i];
      atomicAdd(&sc.nsel, 1);
    }
  }
  __syncthreads();
  if (tid == 0) p.n_left[b] = M - sc.nsel;
  __syncthreads();
}

}  // namespace fdllm
