// Block attention on CUDA cores, one warp per (batch, query, query head).
// Serves fp32 inputs (the tiny fp32 setting) and is the reference-shaped
// fallback for shapes the tensor-core kernel does not cover.  Online softmax
// over 32-key chunks: each lane scores one key, the warp merges (max, sum) with
// shuffles, then the chunk's probabilities are broadcast to accumulate P V with
// the head dimension spread over the lanes.
#include "common.cuh"
#include "internal.h"

namespace fdllm {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int DPL>  // DPL = head_dim / 32 values per lane
__global__ void __launch_bounds__(kWarps * 32)
    attn_simt_kernel(AttnProblem p) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t total = (int64_t)p.batch * p.nq * p.hq;
  if (wid >= total) return;
  const int h = (int)(wid % p.hq);
  const int qi = (int)((wid / p.hq) % p.nq);
  const int b = (int)(wid / ((int64_t)p.hq * p.nq));
  const int kvh = h / (p.hq / p.hkv);
  const int d = p.d;
  const T *q = (const T *)p.q + (((int64_t)b * p.nq + qi) * p.hq + h) * d;
  const T *kc = (const T *)p.kc, *vc = (const T *)p.vc, *kf = (const T *)p.kf, *vf = (const T *)p.vf;

  // scores in log2 units: s = (q . k) * scale * log2(e)
  const float qs = p.scale * kLog2e;
  float m = kNegInf, l = 0.f;
  float acc[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) acc[t] = 0.f;

  auto row = [&](const T *cache, const T *fresh, int j) -> const T * {
    const int f = j - p.fresh0;
    if (f >= 0 && f < p.nq) return fresh + (((int64_t)b * p.nq + f) * p.hkv + kvh) * d;
    return cache + (((int64_t)b * p.seq_len + j) * p.hkv + kvh) * d;
  };

  for (int j0 = 0; j0 < p.seq_len; j0 += 32) {
    const int j = j0 + lane;
    float s = kNegInf;
    if (j < p.seq_len) {
      const T *kr = row(kc, kf, j);
      float dot = 0.f;
      for (int t = 0; t < d; ++t) dot += to_f32(q[t]) * to_f32(kr[t]);
      s = dot * qs;
    }
    float mc = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    const float mn = fmaxf(m, mc);
    const float alpha = (m == kNegInf) ? 0.f : exp2f(m - mn);
    const float pj = (j < p.seq_len) ? exp2f(s - mn) : 0.f;
    float ps = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l = l * alpha + ps;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[t] *= alpha;
    const int nk = min(32, p.seq_len - j0);
    for (int jj = 0; jj < nk; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
      const T *vr = row(vc, vf, j0 + jj);
#pragma unroll
      for (int t = 0; t < DPL; ++t) acc[t] += pb * to_f32(vr[lane + 32 * t]);
    }
    m = mn;
  }
  const float inv = 1.f / l;
  const int64_t ob = (((int64_t)b * p.nq + qi) * p.hq + h) * d;
#pragma unroll
  for (int t = 0; t < DPL; ++t) {
    const float o = acc[t] * inv;
    if (p.out_f32)
      ((float *)p.out)[ob + lane + 32 * t] = o;
    else
      ((T *)p.out)[ob + lane + 32 * t] = from_f32<T>(o);
  }
  if (p.lse && lane == 0)
    p.lse[((int64_t)b * p.nq + qi) * p.hq + h] = (m + log2f(l)) * 0.6931471805599453f;
}

template <typename T>
cudaError_t launch_t(const AttnProblem &p, cudaStream_t st) {
  const int64_t warps = (int64_t)p.batch * p.nq * p.hq;
  const unsigned grid = (unsigned)((warps + kWarps - 1) / kWarps);
  switch (p.d / 32) {
    case 2: attn_simt_kernel<T, 2><<<grid, kWarps * 32, 0, st>>>(p); break;
    case 4: attn_simt_kernel<T, 4><<<grid, kWarps * 32, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t attn_simt_workspace(const AttnProblem &) { return 0; }

cudaError_t launch_attn_simt(const AttnProblem &p, cudaStream_t st) {
  if (p.batch * (int64_t)p.nq * p.hq == 0) return cudaSuccess;
  return p.in_bf16 ? launch_t<__nv_bfloat16>(p, st) : launch_t<float>(p, st);
}

}  // namespace fdllm
