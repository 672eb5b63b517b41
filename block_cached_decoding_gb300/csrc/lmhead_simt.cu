// LM head + online vocabulary reduction on CUDA cores (fp32 inputs, and any
// shape the tensor-core kernel does not take).  Each CTA owns a contiguous
// vocabulary split; each warp walks vocabulary rows of its split in increasing
// order, forms the logits of every masked row with lane-parallel dot products
// and folds them into a per-(warp, row) VocabStat; the warps' states are then
// merged in warp order and written as this split's partial of each masked block
// row (partials [b * B, splits], indexed by block row).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kWarps = 4;
constexpr int kRowGroup = 4;  // masked rows sharing one pass over a W row

// Masked rows of the block in (sequence, position) order, compacted with warp
// ballots; returns the count.  rows[r] = b * B + i.
__device__ int compact_masked_rows(const SelectProblem &p, int *rows) {
  const int32_t *tokens = p.tokens;
  const int batch = p.batch, seq_len = p.seq_len, B = p.B, mask_id = p.mask_id;
  __shared__ int count;
  if (threadIdx.x < 32) {
    int base = 0;
    const int lane = threadIdx.x;
    for (int b = 0; b < batch; ++b) {
      const int sb = seq_block_start(p, b);
      for (int c = 0; c < B; c += 32) {
        const int i = c + lane;
        const bool m = sb >= 0 && i < B && tokens[(int64_t)b * seq_len + sb + i] == mask_id;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (m) rows[base + __popc(bal & ((1u << lane) - 1u))] = b * B + i;
        base += __popc(bal);
      }
    }
    if (lane == 0) count = base;
  }
  __syncthreads();
  return count;
}

template <typename T>
__device__ __forceinline__ void load8(const T *p, float *x);
template <>
__device__ __forceinline__ void load8<float>(const float *p, float *x) {
  const float4 a = *(const float4 *)p, b = *(const float4 *)(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float *x) {
  const uint4 u = *(const uint4 *)p;
  const __nv_bfloat162 *h = (const __nv_bfloat162 *)&u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
    lmhead_simt_kernel(SelectProblem p, VocabStat *__restrict__ part, int splits) {
  extern __shared__ unsigned char smem_raw[];
  int *rows = (int *)smem_raw;                                        // [batch * B]
  VocabStat *st = (VocabStat *)(smem_raw + ((p.batch * p.B * 4 + 15) & ~15));  // [kWarps][R]
  const int R = compact_masked_rows(p, rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tc::pdl_launch_dependents();
  for (int r = threadIdx.x; r < kWarps * R; r += blockDim.x) st[r] = vs_identity();
  __syncthreads();

  const int g = blockIdx.x;
  const int v0 = (int)((int64_t)p.V * g / splits), v1 = (int)((int64_t)p.V * (g + 1) / splits);
  const T *hid = (const T *)p.hidden;
  const T *w = (const T *)p.w;
  for (int v = v0 + warp; v < v1; v += kWarps) {
    const T *wr = w + (int64_t)v * p.H;
    for (int r0 = 0; r0 < R; r0 += kRowGroup) {
      float acc[kRowGroup] = {0.f, 0.f, 0.f, 0.f};
      for (int k = lane * 8; k < p.H; k += 256) {
        float wx[8];
        load8<T>(wr + k, wx);
#pragma unroll
        for (int rr = 0; rr < kRowGroup; ++rr) {
          if (r0 + rr < R) {
            float hx[8];
            load8<T>(hid + (int64_t)rows[r0 + rr] * p.H + k, hx);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[rr] += hx[e] * wx[e];
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < kRowGroup; ++rr) {
        float a = acc[rr];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0 && r0 + rr < R) vs_push(st[warp * R + r0 + rr], a, v);
      }
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    VocabStat acc = st[r];
    for (int w2 = 1; w2 < kWarps; ++w2) acc = vs_merge(acc, st[w2 * R + r]);
    part[(int64_t)rows[r] * splits + g] = acc;  // partials are indexed by block row b * B + i
  }
}

}  // namespace

int lmhead_simt_splits(const SelectProblem &p) {
  int s = sm_count() * 2;
  if (s > p.V) s = p.V;
  return s < 1 ? 1 : s;
}

cudaError_t launch_lmhead_simt(const SelectProblem &p, VocabStat *part, int splits, cudaStream_t st) {
  const size_t smem = (((size_t)p.batch * p.B * 4 + 15) & ~(size_t)15) +
                      (size_t)kWarps * p.batch * p.B * sizeof(VocabStat);
  if (p.in_bf16) {
    auto k = lmhead_simt_kernel<__nv_bfloat16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<splits, kWarps * 32, smem, st>>>(p, part, splits);
  } else {
    auto k = lmhead_simt_kernel<float>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<splits, kWarps * 32, smem, st>>>(p, part, splits);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fdllm
