/*
 * fdllm.h -- C ABI of the GB300 (sm_103a) Fast-dLLM block-cached decoding hot path.
 *
 * Three operations make up one denoising step of block-wise decoding for a
 * masked-diffusion LM ("Fast-dLLM: Training-free Acceleration of Diffusion LLM
 * by Enabling KV Cache and Parallel Decoding", paper-graph-ui summary):
 *
 *   fdllm_block_attn          attention of the recomputed queries over the
 *                             approximate KV cache (section 3.4.2, "PrefixCache"
 *                             and "DualCache"; section 3.4.4 "Cache reuse").
 *   fdllm_confidence_select   LM head over the block's masked positions with an
 *                             online softmax giving confidence and argmax, then
 *                             confidence-aware unmasking (section 3.4.3:
 *                             confidence c_i = max_v p(x_i = v); threshold
 *                             strategy with the progress guarantee; factor
 *                             strategy; the fixed top-k baseline of section 5).
 *   fdllm_kv_splice           writes fresh K/V into the cache window, or the
 *                             whole recomputed cache at a block boundary
 *                             (section 3.4.2 "Cache Overhead and Fused Updates",
 *                             section 3.4.4 step 3 "Cache update").
 *
 * Knob names follow the Fast-dLLM README's command line: gen_length,
 * block_size, use_cache, if_cache_position (here: dual_cache), threshold.
 *
 * Conventions shared by every call
 *  - Pointers marked "device" are CUDA device (or managed) memory owned by the
 *    caller; the library never allocates, frees or retains them.  Every tensor
 *    is dense, row-major in the order its layout names, and 16-byte aligned.
 *  - Calls are asynchronous and ordered on `stream` (NULL: the legacy default
 *    stream).  A returned FDLLM_OK means the work was enqueued.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns FDLLM_EINVAL and launches nothing.  fdllm_last_error()
 *    returns a message for the last failure on the calling thread.
 *  - Kernels never wait without bound.  A device wait that gives up records
 *    FDLLM_ETIMEOUT in a per-device error word, which fdllm_last_device_error()
 *    reads and clears.
 *  - Floating-point inputs are bf16 or fp32 (fdllm_dtype); all accumulation is
 *    fp32.
 */
#ifndef FDLLM_H_
#define FDLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (same type as cudaStream_t / CUstream). */
typedef struct CUstream_st *fdllm_stream_t;

typedef enum {
  FDLLM_OK = 0,
  FDLLM_EINVAL = 1,       /* bad argument: shape, range, alignment, null pointer, small workspace */
  FDLLM_ECUDA = 2,        /* a CUDA runtime call failed (launch error, no device) */
  FDLLM_ETIMEOUT = 3,     /* a bounded device wait expired (see fdllm_last_device_error) */
  FDLLM_EUNSUPPORTED = 4  /* valid request this build does not implement */
} fdllm_status;

typedef enum { FDLLM_BF16 = 0, FDLLM_F32 = 1 } fdllm_dtype;

/* ------------------------------------------------------------------------ */
/* Block attention                                                           */
/* ------------------------------------------------------------------------ */

/* Sequence layout: N = prompt_len + gen_length positions; block k (0-based)
 * spans [s, e) with s = prompt_len + k * block_size, e = s + block_size
 * (section 3.4.4 "Determine block boundaries", written there 1-based).
 *
 * Which positions have fresh (this step's) queries, keys and values:
 *   use_cache = 1, dual_cache = 1  DualCache:   [s, e)   (nq = block_size)
 *   use_cache = 1, dual_cache = 0  PrefixCache: [s, N)   (nq = N - s; block and suffix)
 *   use_cache = 0                  no cache:    [0, N)   (nq = N)
 * Every other position's key and value is read from the cache: the prefix
 * [0, s) and, with DualCache, the suffix [e, N).  Attention is bidirectional
 * (no causal mask): every query attends to all N positions. */
typedef struct {
  int32_t batch;       /* b >= 1 */
  int32_t prompt_len;  /* |p0| >= 0 */
  int32_t gen_length;  /* L >= block_size, a multiple of block_size */
  int32_t block_size;  /* B >= 1 */
  int32_t block_idx;   /* 0 <= k < gen_length / block_size */
  int32_t n_q_heads;   /* Hq, a multiple of n_kv_heads */
  int32_t n_kv_heads;  /* Hkv; query head h reads KV head h / (Hq / Hkv) */
  int32_t head_dim;    /* d: 64 or 128 */
  int32_t use_cache;   /* 0 or 1 */
  int32_t dual_cache;  /* 0 or 1 (ignored when use_cache = 0) */
  float sm_scale;      /* score scale; 0 selects 1 / sqrt(head_dim) */
  int32_t dtype;       /* fdllm_dtype of q, caches and fresh K/V */
  int32_t out_f32;     /* 1: out is fp32; 0: out has `dtype` */
} fdllm_attn_desc;

/* Number of fresh query positions nq for `desc` (see the table above), or -1
 * if the descriptor is invalid. */
int64_t fdllm_attn_query_count(const fdllm_attn_desc *desc);

/* Scratch bytes fdllm_block_attn needs for `desc` (0 for every shape the
 * current kernels take: split-KV partials are merged on chip); 0 on an invalid
 * descriptor. */
size_t fdllm_attn_workspace_size(const fdllm_attn_desc *desc);

/* O_i = sum_j softmax_j(q_i . k_j * sm_scale) v_j over all N positions j.
 *   q        device [b, nq, Hq, d]   fresh queries, positions as in the table
 *   k_cache  device [b, N, Hkv, d]   cached keys (rows at fresh positions unread)
 *   v_cache  device [b, N, Hkv, d]   cached values
 *   k_fresh  device [b, nq, Hkv, d]  this step's keys at the fresh positions
 *   v_fresh  device [b, nq, Hkv, d]  this step's values
 *   out      device [b, nq, Hq, d]   fp32 if out_f32 else dtype
 *   lse      device [b, nq, Hq] fp32 natural-log softmax denominators, or NULL
 *   workspace device, >= fdllm_attn_workspace_size(desc) bytes (NULL if that is 0);
 *            contents on entry are ignored.
 * Errors: FDLLM_EINVAL for an invalid descriptor, a null required pointer, a
 * pointer not 16-byte aligned or a short workspace. */
fdllm_status fdllm_block_attn(const fdllm_attn_desc *desc, const void *q, const void *k_cache,
                              const void *v_cache, const void *k_fresh, const void *v_fresh,
                              void *out, float *lse, void *workspace, size_t ws_bytes,
                              fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* LM head + confidence + parallel unmask                                   */
/* ------------------------------------------------------------------------ */

typedef enum {
  FDLLM_SELECT_THRESHOLD = 0, /* unmask every masked i with c_i > threshold; if none, the single
                                 most confident one (progress guarantee) */
  FDLLM_SELECT_FACTOR = 1,    /* sort by confidence; unmask the largest n with
                                 (n + 1) (1 - c_(n)) < factor, at least one */
  FDLLM_SELECT_TOPK = 2       /* unmask the topk most confident masked positions */
} fdllm_select_strategy;

typedef struct {
  int32_t batch;        /* b >= 1 */
  int32_t seq_len;      /* N, row length of `tokens` */
  int32_t block_start;  /* s: the block is tokens[:, s : s + block_size] */
  int32_t block_size;   /* B, 1..256 */
  int32_t hidden;       /* H, a multiple of 64 */
  int32_t vocab;        /* V >= 2 */
  int32_t mask_id;      /* the [MASK] token id; positions holding it are masked */
  int32_t strategy;     /* fdllm_select_strategy */
  float threshold;      /* tau (strategy THRESHOLD); tau >= 1 unmasks one per step */
  float factor;         /* f > 0 (strategy FACTOR) */
  int32_t topk;         /* k >= 1 (strategy TOPK) */
  int32_t dtype;        /* fdllm_dtype of hidden and lm_head_w */
} fdllm_select_desc;

/* Scratch bytes fdllm_confidence_select needs (a 256-byte header of 8-byte ticket
 * words plus the per-split softmax partials of up to batch * block_size rows); 0 on an invalid
 * descriptor.  The workspace needs no initialisation and may be reused by
 * consecutive calls, but two calls that may run at the same time (different
 * streams) must not share one. */
size_t fdllm_select_workspace_size(const fdllm_select_desc *desc);

/* One confidence-aware unmask step.
 * For every masked position i of the block (tokens[b, s + i] == mask_id) the
 * logits l = hidden[b, i] . W^T are reduced over the whole vocabulary without
 * being stored, giving
 *   argmax[b, i] = lowest v with l_v = max l
 *   conf[b, i]   = c = max_v softmax(l)_v
 *   kappa[b, i]  = log((1 - c) / c), computed without cancellation so it still
 *                  orders positions whose confidence rounds to 1
 * Selection (per `strategy`) ranks by kappa (lowest position first on ties)
 * and writes tokens[b, s + i] = argmax[b, i] for the chosen positions.
 *   hidden        device [b, B, H]   hidden states of all block positions (rows of
 *                                    positions that are not masked are not read)
 *   lm_head_w     device [V, H]      LM-head weight, row v = token v
 *   tokens        device int32 [b, N], updated in place
 *   unmasked      device uint8 [b, B] out: 1 where this step unmasked
 *   conf          device fp32 [b, B] out: c, NaN where not masked
 *   kappa         device fp32 [b, B] out or NULL: log-odds, NaN where not masked
 *   argmax        device int32 [b, B] out: token, -1 where not masked
 *   n_masked_left device int32 [b] out: masked positions left in the block
 *   workspace     device, >= fdllm_select_workspace_size(desc) bytes
 * Errors: FDLLM_EINVAL for an invalid descriptor, null or misaligned pointers, or
 * a short workspace. */
fdllm_status fdllm_confidence_select(const fdllm_select_desc *desc, const void *hidden,
                                     const void *lm_head_w, int32_t *tokens, uint8_t *unmasked,
                                     float *conf, float *kappa, int32_t *argmax,
                                     int32_t *n_masked_left, void *workspace, size_t ws_bytes,
                                     fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Allocation-free confidence select                                         */
/* ------------------------------------------------------------------------ */

/* The paper has no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory, e.g. a plug-in inside a host
 * framework that owns every device allocation and hands the plug-in only its
 * inputs and outputs, or a runtime that forbids allocation once serving has
 * started.  It computes exactly what fdllm_confidence_select computes, with the
 * same arguments except the workspace.
 *
 * Scratch: the per-split vocabulary partials live in a fixed array of
 * FDLLM_NOALLOC_SCRATCH_BYTES (2 MiB) compiled into this library as a
 * file-scope __device__ array; every GPU that loads the library holds it until
 * the process exits.  The call accepts exactly the descriptors for which
 * fdllm_select_workspace_size(desc) <= 2 MiB (for bf16 and batch * block_size
 * <= 512 that is batch * block_size * SM count * 16 bytes); any larger request
 * returns FDLLM_EINVAL with a message and launches nothing.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, so make that first call
 * before any stream capture.
 * Sharing: every call uses the same array and it keeps the last call's
 * contents.  Nothing in it has to start at zero (a call writes every entry it
 * later reads), but calls that overlap on the GPU -- unordered streams, or
 * several host threads -- race on the array and give wrong results; order them
 * on one stream or with events.
 * The call never calls cudaMalloc, cudaFree or any other allocating routine.
 * Errors: as fdllm_confidence_select, plus FDLLM_EINVAL when the partials would
 * exceed the array and FDLLM_ECUDA when the set-up lookup fails. */
#define FDLLM_NOALLOC_SCRATCH_BYTES (2u << 20)

fdllm_status fdllm_confidence_select_noalloc(const fdllm_select_desc *desc, const void *hidden,
                                             const void *lm_head_w, int32_t *tokens,
                                             uint8_t *unmasked, float *conf, float *kappa,
                                             int32_t *argmax, int32_t *n_masked_left,
                                             fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* KV cache splice / refresh                                                 */
/* ------------------------------------------------------------------------ */

typedef enum {
  FDLLM_SPLICE_WINDOW = 0,  /* cache[:, start : start + len] <- src[:, 0 : len] */
  FDLLM_SPLICE_REFRESH = 1  /* block boundary: cache[:, 0 : N] <- src (start must be 0, len = N) */
} fdllm_splice_mode;

/* Copies keys and values into the cache, both as [b, rows, Hkv, d].
 *   k_cache, v_cache  device [b, seq_len, Hkv, d]
 *   k_src, v_src      device [b, len, Hkv, d]
 * Hkv * d * element size must be a multiple of 16 bytes.
 * Errors: FDLLM_EINVAL for a window outside [0, seq_len), REFRESH with
 * start != 0 or len != seq_len, null or misaligned pointers. */
fdllm_status fdllm_kv_splice(int32_t mode, int32_t batch, int32_t seq_len, int32_t n_kv_heads,
                             int32_t head_dim, int32_t start, int32_t len, int32_t dtype,
                             void *k_cache, void *v_cache, const void *k_src, const void *v_src,
                             fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Per-sequence (non-lock-step) blocks                                       */
/* ------------------------------------------------------------------------ */
/* Batched decoding (summary, "Throughput scaling with batch size", Appendix C.5,
 * Figure 9) where each sequence is at its own block: a sequence whose block is
 * done moves to its next block without waiting for the others.  The pages do
 * not describe the batched loop; these calls are the plain per-sequence reading.
 * Each takes the per-sequence block as a device array, so a decode loop can
 * advance it on the GPU.  Indices are checked on the device: a sequence whose
 * index is out of range is skipped and fdllm_last_device_error then reports
 * FDLLM_EINVAL (site 231 select, 232 attention, 233 splice). */

/* fdllm_block_attn with DualCache (desc->dual_cache = 1, use_cache = 1, bf16),
 * sequence b at block block_idx[b] (device int32 [batch], in
 * [0, gen_length / block_size)); desc->block_idx is only validated.  q, k_fresh,
 * v_fresh and out are [b, block_size, H, d] as for fdllm_block_attn.  Rows of
 * sequence b's own window [s_b, s_b + block_size) in the caches may be loaded
 * where a key tile crosses the window's edge, but they never reach the result:
 * their scores are excluded and their values are replaced by zeros before the
 * product, so they may hold anything (NaN and Inf included).  Needs the
 * workspace of fdllm_attn_workspace_size(desc).  FDLLM_EUNSUPPORTED for fp32 or
 * without DualCache. */
fdllm_status fdllm_block_attn_ragged(const fdllm_attn_desc *desc, const int32_t *block_idx, const void *q,
                                     const void *k_cache, const void *v_cache, const void *k_fresh,
                                     const void *v_fresh, void *out, float *lse, void *workspace,
                                     size_t ws_bytes, fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Block attention with the cache-window update                              */
/* ------------------------------------------------------------------------ */
/* The summary's fused cache update (section 3.4.2 "Cache Overhead and Fused
 * Updates"): after a denoising step the block's freshly computed keys and
 * values replace the cache window, and writing them from the attention call
 * itself -- which has just read them -- saves the separate copy and its re-read.
 *
 * fdllm_block_attn (block_idx NULL) or fdllm_block_attn_ragged (block_idx
 * non-NULL, DualCache) plus, for every sequence b, cache rows [s_b, s_b +
 * block_size) <- the first block_size fresh rows (k_fresh / v_fresh rows 0 ..
 * block_size - 1, the block), exactly as fdllm_kv_splice(FDLLM_SPLICE_WINDOW,
 * ..., s_b, block_size) would after the attention.  The attention reads no cache
 * row of the window (DualCache reads the block's fresh keys there; PrefixCache
 * reads only [0, s)), so the result equals the two separate calls.  Arguments
 * and errors as fdllm_block_attn; k_cache and v_cache are written.  Requires
 * use_cache = 1 (else FDLLM_EUNSUPPORTED).  When the kernel cannot store the
 * window itself -- the block does not fill whole key tiles of its plan, or fp32
 * inputs -- a DualCache call with block_idx NULL launches the splice kernel after
 * the attention (two kernels); per-sequence blocks and PrefixCache then return
 * FDLLM_EUNSUPPORTED. */
fdllm_status fdllm_block_attn_update(const fdllm_attn_desc *desc, const int32_t *block_idx, const void *q,
                                     void *k_cache, void *v_cache, const void *k_fresh, const void *v_fresh,
                                     void *out, float *lse, void *workspace, size_t ws_bytes,
                                     fdllm_stream_t stream);

/* fdllm_confidence_select with sequence b's block starting at block_start[b]
 * (device int32 [batch], in [0, seq_len - block_size]); desc->block_start is
 * only validated.  Same workspace (fdllm_select_workspace_size(desc)) and
 * outputs; hidden row (b, i) is the state of position block_start[b] + i. */
fdllm_status fdllm_confidence_select_ragged(const fdllm_select_desc *desc, const int32_t *block_start,
                                            const void *hidden, const void *lm_head_w, int32_t *tokens,
                                            uint8_t *unmasked, float *conf, float *kappa, int32_t *argmax,
                                            int32_t *n_masked_left, void *workspace, size_t ws_bytes,
                                            fdllm_stream_t stream);

/* FDLLM_SPLICE_WINDOW with sequence b's window at start[b] (device int32
 * [batch], in [0, seq_len - len]): cache[b, start[b] : start[b] + len] <- src[b]. */
fdllm_status fdllm_kv_splice_ragged(int32_t batch, int32_t seq_len, int32_t n_kv_heads, int32_t head_dim,
                                    const int32_t *start, int32_t len, int32_t dtype, void *k_cache,
                                    void *v_cache, const void *k_src, const void *v_src, fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* FP8 weight cache                                                          */
/* ------------------------------------------------------------------------ */
/* The summary proposes FP8 or INT8 storage for cached activations as future
 * work (section 6, the memory-overhead limitation; section 7, future direction
 * 3 "KV cache quantization and memory-efficient DualCache") without a scheme.
 * Here the LM-head weight, the largest per-step read of the path, is stored in
 * FP8: E4M3 codes (OCP FP8: bias 7, 3 mantissa bits, subnormals, largest finite
 * value 448) with one power-of-two scale per row.  Row r's scale is 2^k, k the
 * smallest integer with max|row| <= 448 * 2^k (k = 0 for an all-zero row), and
 * its codes are x / 2^k rounded to the nearest E4M3 value, ties to even.  Inputs
 * must be finite. */

/* q[r, :] (uint8 E4M3 codes, device [rows, cols]) and scale[r] (device float
 * [rows]) for each row of src (device [rows, cols], `dtype`).  Asynchronous on
 * `stream`; returns FDLLM_EINVAL for a negative shape, a bad dtype or a null
 * pointer (nothing to do for rows = 0 or cols = 0). */
fdllm_status fdllm_quantize_fp8_rows(int64_t rows, int32_t cols, int32_t dtype, const void *src, uint8_t *q,
                                     float *scale, fdllm_stream_t stream);

/* Workspace bytes of fdllm_confidence_select_fp8w (the select workspace plus
 * the block's hidden rows in E4M3 and their scales); 0 on an invalid or
 * unsupported descriptor. */
size_t fdllm_select_fp8w_workspace_size(const fdllm_select_desc *desc);

/* fdllm_confidence_select with the LM-head weight from the FP8 cache: w_q
 * (device uint8 [V, H]) and w_scale (device float [V]) as written by
 * fdllm_quantize_fp8_rows.  The block's hidden rows (bf16, desc->dtype =
 * FDLLM_BF16) are quantised the same way, per row, into the workspace, and
 * logit l_v = h_scale * w_scale[v] * sum_k qh_k qw_vk (fp32 accumulation); the
 * reduction, selection and outputs are those of fdllm_confidence_select.
 * FDLLM_EUNSUPPORTED unless hidden is a multiple of 128 and batch * block_size
 * <= 512.  Two kernels per call. */
fdllm_status fdllm_confidence_select_fp8w(const fdllm_select_desc *desc, const void *hidden, const uint8_t *w_q,
                                          const float *w_scale, int32_t *tokens, uint8_t *unmasked, float *conf,
                                          float *kappa, int32_t *argmax, int32_t *n_masked_left, void *workspace,
                                          size_t ws_bytes, fdllm_stream_t stream);

/* FP8 KV cache (the summary's future direction 3).  Cached keys and values
 * are stored per (sequence, position, KV head) row of head_dim values by the
 * rule above: k_cache / v_cache hold E4M3 codes (device uint8 [b, N, Hkv, d])
 * and k_scale / v_scale the row scales (device float [b, N, Hkv]).  Queries
 * and this step's fresh keys and values stay bf16. */

/* fdllm_block_attn (or, with block_idx non-NULL, fdllm_block_attn_ragged) over
 * an FP8 cache: the result is the attention over the dequantised cache
 * (code * scale, exact in bf16).  desc->dtype must be FDLLM_BF16 and
 * desc->use_cache 1 (PrefixCache or DualCache), else FDLLM_EUNSUPPORTED; null
 * scales give FDLLM_EINVAL.  Cache rows at the fresh positions (codes and
 * scales) may be loaded where a key tile crosses a range edge but never reach
 * the result (their keys and values are replaced by zeros), so they may hold
 * anything. */
fdllm_status fdllm_block_attn_fp8kv(const fdllm_attn_desc *desc, const int32_t *block_idx, const void *q,
                                   const uint8_t *k_cache, const float *k_scale, const uint8_t *v_cache,
                                   const float *v_scale, const void *k_fresh, const void *v_fresh, void *out,
                                   float *lse, void *workspace, size_t ws_bytes, fdllm_stream_t stream);

/* fdllm_kv_splice into an FP8 cache: each source row (b, i, h) of head_dim
 * values (src [b, len, Hkv, d], `src_dtype` bf16 or fp32) is quantised into
 * cache row (b, start + i, h) and its scale; every other row is unchanged.
 * Modes and window checks as for fdllm_kv_splice.  Two kernels per call. */
fdllm_status fdllm_kv_splice_fp8(int32_t mode, int32_t batch, int32_t seq_len, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t start, int32_t len, int32_t src_dtype,
                                 uint8_t *k_cache, float *k_scale, uint8_t *v_cache, float *v_scale,
                                 const void *k_src, const void *v_src, fdllm_stream_t stream);

/* The window splice into an FP8 cache with sequence b's window at start[b]
 * (device int32 [batch], in [0, seq_len - len]; a start outside it skips the
 * sequence and sets device error site 233, as fdllm_kv_splice_ragged does). */
fdllm_status fdllm_kv_splice_fp8_ragged(int32_t batch, int32_t seq_len, int32_t n_kv_heads, int32_t head_dim,
                                        const int32_t *start, int32_t len, int32_t src_dtype, uint8_t *k_cache,
                                        float *k_scale, uint8_t *v_cache, float *v_scale, const void *k_src,
                                        const void *v_src, fdllm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Device-driven block loop                                                  */
/* ------------------------------------------------------------------------ */
/* The block loop of Algorithm 1 (summary 3.4.4) repeats denoising steps until
 * the block has no mask; a host-driven loop reads the masked count back after
 * every step (the pages' PyTorch form synchronises on it).  This executor runs
 * the repetition on the device: `step` is called once, with a capture stream,
 * and must enqueue one whole denoising step on it (the step's inputs, the
 * attention, fdllm_confidence_select writing n_masked_left, any splice); that
 * work becomes the body of a CUDA graph while-loop, and a control kernel after
 * it counts the step in *step_counter (device int64; 0 at the start of each
 * launch) and, if total_steps is not NULL, in *total_steps (device int64,
 * never reset: a running step index across launches); captured work may read
 * either to key per-step inputs.  It repeats
 * the body while some n_masked_left[b] > 0 (b < batch) and fewer than
 * max_steps steps have run.  The body always runs at least once.  Pointers and
 * descriptors are captured by value: each launch re-runs the same calls on the
 * same buffers.  Capture uses relaxed mode; `step` must not synchronise.
 * Kernels launched by the graph are not added to fdllm_launch_counter. */
typedef struct fdllm_block_loop fdllm_block_loop;
typedef void (*fdllm_step_fn)(void *user, fdllm_stream_t stream);

/* Build and instantiate the loop; FDLLM_EINVAL for null pointers, batch < 1
 * or max_steps < 1, FDLLM_ECUDA if capture or instantiation fails. */
fdllm_status fdllm_block_loop_create(fdllm_block_loop **loop, fdllm_step_fn step, void *user,
                                     const int32_t *n_masked_left, int32_t batch, int32_t max_steps,
                                     int64_t *step_counter, int64_t *total_steps);

/* The same loop with the cache refreshed every `refresh_every` steps inside the
 * block (the summary's refresh-every-r-steps cache, section 5 Table 10, reported
 * for LLaDA-V): `refresh` is called once, with a capture stream, and must enqueue
 * the refresh (the recomputed caches written with FDLLM_SPLICE_REFRESH); it runs
 * on the device before step c of a launch whenever c > 0 and refresh_every
 * divides c (the caller refreshes before step 0, at the block boundary).
 * Captured work may read *step_counter (step c of the block) to key the refresh.
 * FDLLM_EINVAL for refresh_every < 1 or a null refresh, else as
 * fdllm_block_loop_create. */
fdllm_status fdllm_block_loop_create_refresh(fdllm_block_loop **loop, fdllm_step_fn step, fdllm_step_fn refresh,
                                             void *user, const int32_t *n_masked_left, int32_t batch,
                                             int32_t max_steps, int32_t refresh_every, int64_t *step_counter,
                                             int64_t *total_steps);

/* A whole generation in the per-sequence regime as one device-driven loop
 * (Fast-dLLM summary §5 "Throughput scaling with batch size" and Appendix
 * C.5: each sequence of the batch moves to its next block as soon as its own
 * block has no mask, rather than waiting for the whole batch).  The caller's
 * `step` reads the per-sequence state below (typically through the *_ragged
 * calls: block_idx for the attention, block_start for the select and splice)
 * and writes n_masked_left.  After each step the control kernel, for every
 * unfinished sequence b: adds 1 to seq_steps[b]; if n_masked_left[b] is 0,
 * either moves it to its next block (block_idx[b] += 1, block_start[b] +=
 * block_size, refresh_flags[b] = 1) or, after block n_blocks - 1, sets
 * done[b] = 1.  refresh_flags of sequences that did not move are cleared.
 * The loop repeats while some done[b] is 0 and fewer than max_steps steps
 * have run (n_blocks * block_size always suffices: every step unmasks at
 * least one position of every unfinished sequence).  With a non-null
 * `refresh`, it is captured into a conditional node that runs before the next
 * step whenever some sequence moved: it should recompute the caches of the
 * flagged sequences (reading refresh_flags and block_idx).  A finished
 * sequence keeps its last block index, so the captured calls stay in range;
 * it has no masked position left, so its outputs no longer change.
 *
 * Arguments (all device memory, int32 / uint8 [batch], caller-initialised
 * before each launch: block_idx the first block of each sequence, block_start
 * = prompt_len + block_idx * block_size, seq_steps 0, refresh_flags 0, done 0,
 * and the caches refreshed for the first blocks): as listed; step_counter /
 * total_steps as in fdllm_block_loop_create (steps of this launch / all
 * launches).  FDLLM_EINVAL for a null state pointer, batch < 1,
 * n_blocks < 1, block_size < 1 or max_steps < 1; FDLLM_ECUDA if capture or
 * instantiation fails. */
fdllm_status fdllm_block_loop_create_ragged(fdllm_block_loop **loop, fdllm_step_fn step, fdllm_step_fn refresh,
                                            void *user, const int32_t *n_masked_left, int32_t batch,
                                            int32_t n_blocks, int32_t block_size, int32_t max_steps,
                                            int32_t *block_idx, int32_t *block_start, int32_t *seq_steps,
                                            uint8_t *refresh_flags, uint8_t *done, int64_t *step_counter,
                                            int64_t *total_steps);

/* Run the loop once on `stream` (asynchronous). */
fdllm_status fdllm_block_loop_launch(fdllm_block_loop *loop, fdllm_stream_t stream);

void fdllm_block_loop_destroy(fdllm_block_loop *loop);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Static description of a status code. */
const char *fdllm_status_string(int32_t status);

/* Message describing the last non-OK status returned on the calling thread
 * (thread-local; valid until the next failing call on that thread). */
const char *fdllm_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's error
 * word: FDLLM_OK if nothing was recorded since the last read; FDLLM_EINVAL if a
 * per-sequence block index was out of range (sites 231-233); else FDLLM_ETIMEOUT,
 * a device wait that gave up (`detail`, if not NULL, receives the site code). */
fdllm_status fdllm_last_device_error(fdllm_stream_t stream, int32_t *detail);

/* Failure-detection self-test: launches one CTA that waits, through the same
 * bounded mbarrier wait the kernels use, on a barrier nothing ever arrives at,
 * with a limit of `limit_ms` milliseconds (1..1000).  The wait gives up,
 * records site code 900 in the device error word and the kernel returns, so
 * fdllm_last_device_error then reports FDLLM_ETIMEOUT and the CUDA context stays
 * usable.  Returns FDLLM_EINVAL for a limit outside 1..1000. */
fdllm_status fdllm_selftest_bounded_wait(int32_t limit_ms, fdllm_stream_t stream);

/* ABI version: 100 * major + minor (101: the per-sequence block calls; 102: the
 * FP8 weight cache; 103: the FP8 KV cache; 104: the device-driven block loop;
 * 105: fdllm_block_attn_update and the loop's refresh every r steps; 106: the
 * per-sequence device-driven loop). */
int32_t fdllm_version(void);

/* Number of kernels this library has launched in the process so far (all
 * devices, all threads): a diagnostic for counting launches per step. */
uint64_t fdllm_launch_counter(void);

#ifdef __cplusplus
}
#endif

#endif /* FDLLM_H_ */
