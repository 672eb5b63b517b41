// Shared device helpers for the fdllm kernels (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fdllm.h"

namespace fdllm {

#define kNegInf (-__int_as_float(0x7f800000))

// ---------------------------------------------------------------------------
// Element access for the two storage types.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// Online vocabulary reduction state for one row of logits over a set S of ids:
//   m1 = max_{v in S} l_v, a1 = lowest v attaining it,
//   m2 = max_{v in S, v != a1} l_v, s2 = sum_{v in S, v != a1} exp(l_v - m2).
// Then c = 1 / (1 + exp(kappa)) with kappa = (m2 - m1) + log(s2), which stays
// finite (and ordered) when c rounds to 1.  Merging is associative and
// commutative up to rounding; the winner rule (larger m1, then lower id) makes
// a1 independent of the merge order.
// ---------------------------------------------------------------------------
struct __align__(16) VocabStat {
  float m1;
  int32_t a1;
  float m2;
  float s2;
};

__device__ __forceinline__ VocabStat vs_identity() {
  VocabStat s;
  s.m1 = kNegInf;
  s.a1 = 0x7fffffff;
  s.m2 = kNegInf;
  s.s2 = 0.f;
  return s;
}

// s2 * exp(m - ref), with empty sets (s2 == 0) contributing 0 even at m = -inf.
__device__ __forceinline__ float vs_rescale(float s2, float m, float ref) {
  return s2 == 0.f ? 0.f : s2 * __expf(m - ref);
}

__device__ __forceinline__ VocabStat vs_merge(VocabStat a, VocabStat b) {
  const bool b_wins = (b.m1 > a.m1) || (b.m1 == a.m1 && b.a1 < a.a1);
  const VocabStat w = b_wins ? b : a;
  const VocabStat l = b_wins ? a : b;
  VocabStat r;
  r.m1 = w.m1;
  r.a1 = w.a1;
  const float m2 = fmaxf(w.m2, l.m1);  // l.m1 >= l.m2
  r.m2 = m2;
  if (m2 == kNegInf) {
    r.s2 = 0.f;
  } else {
    const float lone = (l.m1 == kNegInf) ? 0.f : __expf(l.m1 - m2);
    r.s2 = vs_rescale(w.s2, w.m2, m2) + lone + vs_rescale(l.s2, l.m2, m2);
  }
  return r;
}

// Add one logit `x` with id `v`; ids arrive in increasing order within a thread,
// so an equal logit never displaces the current argmax.
__device__ __forceinline__ void vs_push(VocabStat &s, float x, int32_t v) {
  if (x > s.m1) {
    if (s.m1 != kNegInf) {  // the old maximum joins the rest
      s.s2 = vs_rescale(s.s2, s.m2, s.m1) + 1.f;
      s.m2 = s.m1;
    }
    s.m1 = x;
    s.a1 = v;
  } else if (x > s.m2) {
    s.s2 = vs_rescale(s.s2, s.m2, x) + 1.f;
    s.m2 = x;
  } else {
    s.s2 += __expf(x - s.m2);
  }
}

// Statistics of 32 logits x[e] with ids v0 + e (in increasing order), without data-dependent
// branches: a pairwise tree of (max, lowest id of the max, second value) over adjacent ranges --
// the left range holds the lower ids, so it wins ties -- then the 31 other terms' exponentials
// relative to the second value, summed as a tree.  Entries of -inf (ids past the vocabulary) never
// win unless all are -inf, which gives the empty statistics.
__device__ __forceinline__ VocabStat vs_chunk32(const float (&x)[32], int32_t v0) {
  float m1[16], m2[16];
  int i1[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const bool ge = x[2 * e] >= x[2 * e + 1];
    m1[e] = ge ? x[2 * e] : x[2 * e + 1];
    m2[e] = ge ? x[2 * e + 1] : x[2 * e];
    i1[e] = ge ? 2 * e : 2 * e + 1;
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
    for (int e = 0; e < w; ++e) {   // node e <- nodes 2e (lower ids) and 2e + 1
      const bool ge = m1[2 * e] >= m1[2 * e + 1];
      const float a2 = fmaxf(m2[2 * e], m1[2 * e + 1]), b2 = fmaxf(m2[2 * e + 1], m1[2 * e]);
      m1[e] = ge ? m1[2 * e] : m1[2 * e + 1];
      i1[e] = ge ? i1[2 * e] : i1[2 * e + 1];
      m2[e] = ge ? a2 : b2;
    }
  }
  VocabStat c;
  c.m1 = m1[0];
  c.a1 = c.m1 == kNegInf ? 0x7fffffff : v0 + i1[0];
  c.m2 = m2[0];
  float t[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) t[e] = e == i1[0] ? 0.f : __expf(x[e] - c.m2);
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) t[e] += t[e + w];
  c.s2 = c.m2 == kNegInf ? 0.f : t[0];
  return c;
}

__device__ __forceinline__ VocabStat vs_shfl_xor(const VocabStat &s, int mask) {
  VocabStat o;
  o.m1 = __shfl_xor_sync(0xffffffffu, s.m1, mask);
  o.a1 = __shfl_xor_sync(0xffffffffu, s.a1, mask);
  o.m2 = __shfl_xor_sync(0xffffffffu, s.m2, mask);
  o.s2 = __shfl_xor_sync(0xffffffffu, s.s2, mask);
  return o;
}

// kappa = log((1 - c) / c) from a complete state.
__device__ __forceinline__ float vs_kappa(const VocabStat &s) {
  if (s.s2 == 0.f) return kNegInf;  // a one-token vocabulary
  return (s.m2 - s.m1) + __logf(s.s2);
}

// ---------------------------------------------------------------------------
// Bounded device waits that give up record a site code in the per-device error
// word (owned by api.cu, passed to kernels as a pointer); the first code wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_device_error(int32_t *err, int32_t site) {
  if (err != nullptr) atomicCAS(err, 0, site);
}

}  // namespace fdllm
