// Merge of the per-split vocabulary partials of one sequence's masked rows into
// confidence / log-odds / argmax, then the unmask decision for its block.
// Shared by select_kernel (one CTA per sequence) and the tail of the
// tensor-core LM-head kernel (its last CTAs to arrive take the sequences once
// every CTA's partials are written).
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
constexpr int kSelectBatchedSplitsPerLane = 5;  // splits <= 160: several rows' loads in flight at once

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
  int mpos[kSelectMaxBlock];   // masked positions in increasing order
  float kapc[kSelectMaxBlock]; // kappa of the j-th masked position
  float kap[kSelectMaxBlock];
  float cf[kSelectMaxBlock];
  int tok[kSelectMaxBlock];
  int m, any, nbest, nsel, start;
};

// The merged statistics of the j-th masked position into the scratch (lane 0 of the merging warp).
__device__ __forceinline__ void store_row(SelectScratch &sc, int j, const VocabStat &acc) {
  const int i = sc.mpos[j];
  const float k = vs_kappa(acc);
  sc.kapc[j] = k;
  sc.kap[i] = k;
  sc.cf[i] = 1.f / (1.f + __expf(k));
  sc.tok[i] = acc.a1;
}

// The two phases below are called by all NT threads of the CTA (NT >= block
// size, a multiple of 32).  select_prepare reads only the tokens (an input):
// this sequence's masked positions, in order, and a cleared scratch.  A caller
// that has already compared every block row's token with the mask id passes
// those flags (`masked`, shared memory, indexed by b * B + i), and the tokens
// are not read again.
template <int NT>
__device__ __forceinline__ void select_prepare(const SelectProblem &p, int b, SelectScratch &sc,
                                               const uint8_t *masked = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B;
  const int sb = seq_block_start(p, b);
  const int32_t *trow = p.tokens + (int64_t)b * p.seq_len + (sb < 0 ? 0 : sb);
  if (tid == 0) {
    sc.any = 0; sc.nbest = 0; sc.nsel = 0; sc.start = sb;
    if (sb < 0) record_device_error(p.err, 231);
  }
  if (warp == 0) {
    int base = 0;
    for (int c = 0; c < B; c += 32) {
      const int i = c + lane;
      const bool m = sb >= 0 && i < B && (masked ? masked[b * B + i] != 0 : trow[i] == p.mask_id);
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
}

// select_finish (after select_prepare for the same b and scratch): `part` holds
// the VocabStat partials [b * B + i][splits]; each masked row of sequence b is
// merged by one warp with a fixed reduction tree (lane-strided partials in
// increasing split order, then an xor butterfly), so the result does not
// depend on which warp or how many rows at a time; then the selection rule and
// the outputs.
template <int NT>
__device__ __forceinline__ void select_finish(const SelectProblem &p, const VocabStat *__restrict__ part,
                                              int splits, int b, SelectScratch &sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NT / 32;
  const int B = p.B;
  const int M = sc.m;

  const VocabStat *__restrict__ pseq = part + (int64_t)b * B * splits;
  if (splits <= 32 * kSelectBatchedSplitsPerLane) {
    // R rows per warp per round; every load is issued before the first use, and each row is
    // reduced in three flat passes (no chain of pairwise merges):
    //   (M1, A1) = the largest m1, lowest id on ties;
    //   M2 = the largest value other than the winner: every m2, and every other split's m1;
    //   S = sum of s2 e^(m2 - M2) over all splits + e^(m1 - M2) over the other splits;
    // then kappa = (M2 - M1) + log S.  Lane-strided partials in increasing split order, then
    // an xor butterfly: the result does not depend on which warp or how many rows at a time.
    constexpr int R = NT <= 256 ? 4 : 2;
    constexpr int KP = kSelectBatchedSplitsPerLane;
    for (int j0 = warp; j0 < M; j0 += NW * R) {
      VocabStat v[R][KP];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = j0 + r * NW;
        const VocabStat *pr = pseq + (int64_t)(j < M ? sc.mpos[j] : 0) * splits;
#pragma unroll
        for (int k = 0; k < KP; ++k) {
          const int gi = lane + 32 * k;
          v[r][k] = (j < M && gi < splits) ? pr[gi] : vs_identity();
        }
      }
      float m1[R], m2[R], sum[R];
      int a1[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        m1[r] = kNegInf;
        a1[r] = 0x7fffffff;
#pragma unroll
        for (int k = 0; k < KP; ++k) {
          const bool w = v[r][k].m1 > m1[r] || (v[r][k].m1 == m1[r] && v[r][k].a1 < a1[r]);
          m1[r] = w ? v[r][k].m1 : m1[r];
          a1[r] = w ? v[r][k].a1 : a1[r];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float om = __shfl_xor_sync(0xffffffffu, m1[r], o);
          const int oa = __shfl_xor_sync(0xffffffffu, a1[r], o);
          const bool w = om > m1[r] || (om == m1[r] && oa < a1[r]);
          m1[r] = w ? om : m1[r];
          a1[r] = w ? oa : a1[r];
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        m2[r] = kNegInf;
#pragma unroll
        for (int k = 0; k < KP; ++k)
          m2[r] = fmaxf(m2[r], fmaxf(v[r][k].m2, v[r][k].a1 == a1[r] ? kNegInf : v[r][k].m1));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) m2[r] = fmaxf(m2[r], __shfl_xor_sync(0xffffffffu, m2[r], o));
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        sum[r] = 0.f;
        if (m2[r] != kNegInf) {
#pragma unroll
          for (int k = 0; k < KP; ++k) {
            if (v[r][k].s2 != 0.f) sum[r] += v[r][k].s2 * __expf(v[r][k].m2 - m2[r]);
            if (v[r][k].a1 != a1[r] && v[r][k].m1 != kNegInf) sum[r] += __expf(v[r][k].m1 - m2[r]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], o);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = j0 + r * NW;
        if (lane == 0 && j < M) {
          VocabStat acc;
          acc.m1 = m1[r]; acc.a1 = a1[r]; acc.m2 = m2[r]; acc.s2 = sum[r];
          store_row(sc, j, acc);
        }
      }
    }
  } else {
    for (int j = warp; j < M; j += NW) {
      const VocabStat acc = merge_row(pseq + (int64_t)sc.mpos[j] * splits, splits);
      if (lane == 0) store_row(sc, j, acc);
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
#pragma unroll 8
      for (int j = 0; j < M; ++j) {
        const float kj = sc.kapc[j];
        const int pj = sc.mpos[j];
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
      p.tokens[(int64_t)b * p.seq_len + sc.start + i] = sc.tok[i];
      atomicAdd(&sc.nsel, 1);
    }
  }
  __syncthreads();
  if (tid == 0) p.n_left[b] = M - sc.nsel;
  __syncthreads();
}

// Both phases for sequence b.
template <int NT>
__device__ __forceinline__ void select_sequence(const SelectProblem &p, const VocabStat *__restrict__ part,
                                                int splits, int b, SelectScratch &sc,
                                                const uint8_t *masked = nullptr) {
  select_prepare<NT>(p, b, sc, masked);
  select_finish<NT>(p, part, splits, b, sc);
}

}  // namespace fdllm
