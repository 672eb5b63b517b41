// Launchers shared between the host ABI (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fdllm.h"

namespace fdllm {

struct VocabStat;  // common.cuh

// Resolved attention problem (validated by api.cu).
struct AttnProblem {
  int batch, seq_len, nq, hq, hkv, d;
  int fresh0;       // first position with fresh K/V (== first query position)
  // per-sequence DualCache blocks (null: every sequence at fresh0): sequence b's block is
  // blocks[b], its window [prompt_len + blocks[b] * nq, + nq); nblocks bounds the index
  const int32_t *blocks;
  int prompt_len, nblocks;
  float scale;      // softmax scale
  int in_bf16;      // q / k / v storage
  // FP8 KV cache (f8kv = 1): kc / vc hold E4M3 codes [b, N, Hkv, d] with scales [b, N, Hkv]
  int f8kv;
  const float *k_scale, *v_scale;
  int out_f32;
  // cache-window update fused into the call (update = 1): cache rows [s, s + win) of each sequence <-
  // the first `win` fresh rows; kc_w / vc_w are the caches, writable
  int update, win;
  void *kc_w, *vc_w;
  const void *q, *kc, *vc, *kf, *vf;
  void *out;
  float *lse;
  void *ws;
  size_t ws_bytes;
  int32_t *err;
};

// Resolved select problem.
struct SelectProblem {
  int batch, seq_len, s, B, H, V, mask_id, strategy, topk;
  const int32_t *starts;  // device [batch]: sequence b's block starts at starts[b] (null: every block at s)
  float kappa_tau;  // c > tau  <=>  kappa < kappa_tau
  float factor;
  int in_bf16;
  const void *hidden, *w;
  // FP8 weight cache (fp8w = 1): w holds E4M3 codes [V, H] with w_scale [V]; the hidden rows are
  // quantised per row into hq [b * B, H] (E4M3) with h_scale [b * B] before the LM head, or, with
  // quant_hidden, by the LM-head kernel itself (both in the workspace)
  int fp8w, quant_hidden;
  const float *w_scale, *h_scale;
  const void *hq;
  int32_t *tokens;
  uint8_t *unmasked;
  float *conf, *kappa;
  int32_t *argmax, *n_left;
  void *ws;
  size_t ws_bytes;
  int32_t *err;
};

#ifdef __CUDACC__
// Block start of sequence b: its own when the problem gives one per sequence, else the shared one;
// -1 when a per-sequence start does not fit the sequence (the select records device error 231).
__device__ __forceinline__ int seq_block_start(const SelectProblem &p, int b) {
  if (p.starts == nullptr) return p.s;
  const int v = p.starts[b];
  return (v >= 0 && v <= p.seq_len - p.B) ? v : -1;
}
#endif

int sm_count();  // SMs of the current device (cached per device)
void count_launches(int n);  // adds to fdllm_launch_counter()

// attn_simt.cu
size_t attn_simt_workspace(const AttnProblem &p);
cudaError_t launch_attn_simt(const AttnProblem &p, cudaStream_t st);

// attn_tc.cu: tcgen05 block attention (bf16, head_dim 64 / 128)
bool attn_tc_supported(const AttnProblem &p);
size_t attn_tc_workspace(const AttnProblem &p);
cudaError_t launch_attn_tc(const AttnProblem &p, cudaStream_t st);
// whether launch_attn_tc stores the cache window itself for p (p.update): the block's rows must fill
// whole key tiles of the kernel's plan, or be a single head's rows within one tile
bool attn_tc_fuses_update(const AttnProblem &p);

// lmhead_simt.cu: per-split vocabulary partials for the masked rows
int lmhead_simt_splits(const SelectProblem &p);
cudaError_t launch_lmhead_simt(const SelectProblem &p, VocabStat *part, int splits, cudaStream_t st);

// lmhead_tc.cu: the tcgen05 kernel (bf16, batch * B <= 512) writes the partials
// [b * B, splits] and runs the merge + select itself; `ticket` is 8 bytes of
// workspace.  lmhead_tc_grid gives the number of vocabulary splits (clusters).
bool lmhead_tc_supported(const SelectProblem &p);
// true when the kernel runs in thread-block clusters (more than 128 block rows): its operand tiles
// are then multicast between the CTAs of a cluster, and the operands must be device memory of the
// current device
bool lmhead_tc_clustered(const SelectProblem &p);
int lmhead_tc_grid(const SelectProblem &p);
bool lmhead_tc_quantises_hidden(const SelectProblem &p);
cudaError_t launch_lmhead_tc(const SelectProblem &p, VocabStat *part, unsigned long long *ticket, int splits,
                             cudaStream_t st);

// fp8.cu: per-row E4M3 quantisation q [rows, cols], scale [rows] of a bf16 / fp32 matrix (the
// rounding and scale rule of the FP8 weight cache); programmatic-dependent launch
cudaError_t launch_quantize_fp8(const void *src, bool src_bf16, int64_t rows, int cols, uint8_t *q, float *scale,
                                cudaStream_t st);
// batch groups of rpb rows: source row bb * src_bstride + r -> codes / scale row bb * dst_bstride + r,
// plus starts[bb] * row_step with a per-sequence start array (device; a start outside [0, max_start]
// skips the sequence and records device error 233 in err)
cudaError_t launch_quantize_fp8_batched(const void *src, bool src_bf16, int64_t batch, int64_t rpb, int cols,
                                        int64_t src_bstride, uint8_t *q, float *scale, int64_t dst_bstride,
                                        cudaStream_t st, const int32_t *starts = nullptr, int64_t row_step = 0,
                                        int max_start = 0, int32_t *err = nullptr);

// select.cu: merge partials [b * B, splits] over splits and unmask
cudaError_t launch_select(const SelectProblem &p, const VocabStat *part, int splits, cudaStream_t st);

// splice.cu: cache[b, start_b : start_b + len] <- src[b] for K and V, start_b = starts[b] when
// `starts` (device) is given, else `start`; a start outside [0, cache_rows - len] skips the sequence
// and records device error 233 in `err`
cudaError_t launch_splice(int batch, int64_t cache_rows, int64_t row_bytes, int64_t start,
                          int64_t len, void *kc, void *vc, const void *ks, const void *vs,
                          cudaStream_t st, const int32_t *starts = nullptr, int32_t *err = nullptr);

}  // namespace fdllm
