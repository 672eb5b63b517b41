/*
 * fdllm_synth.h -- device-side twin of the seeded synthetic input generator.
 *
 * Not part of the decoding method: these calls fill device buffers with the
 * same bytes as the numpy generator (block_cached_decoding_gb300/synth.py), so
 * benchmarks and full-size tests can draw inputs on the GPU.  Both sides
 * implement SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) and the Irwin-Hall
 * "sum of twelve uniforms minus six" normal deviate with exact integer
 * arithmetic, one float32 multiply by sigma (round to nearest even) and
 * round-to-nearest-even conversion to bf16.  Stream keys chain coordinates:
 * key = seed; for each coordinate c: key = splitmix(key, c).
 *
 * All output pointers are caller-owned device memory; calls are asynchronous on
 * `stream`.  Return value: an fdllm_status (0 = OK, 1 = bad argument, 2 = CUDA
 * error).
 */
#ifndef FDLLM_SYNTH_H_
#define FDLLM_SYNTH_H_

#include <stdint.h>

#include "fdllm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Tensor kinds (first coordinate of every stream key). */
enum {
  FDLLM_SYNTH_W = 1,
  FDLLM_SYNTH_KCACHE = 2,
  FDLLM_SYNTH_VCACHE = 3,
  FDLLM_SYNTH_Q = 4,
  FDLLM_SYNTH_KFRESH = 5,
  FDLLM_SYNTH_VFRESH = 6,
  FDLLM_SYNTH_HID = 7,
  FDLLM_SYNTH_PLANT = 8,
  FDLLM_SYNTH_PROMPT = 9
};

/* out[i] = sigma * z(key(seed, coords...), offset + i) for i < n, stored as `dtype`.
 * n_coords <= 4 integer coordinates follow `kind`. */
int32_t fdllm_synth_normals(uint64_t seed, int32_t kind, const int64_t *coords, int32_t n_coords,
                            int64_t n, int64_t offset, float sigma, int32_t dtype, void *out,
                            fdllm_stream_t stream);

/* Cache of one refresh epoch: out [b, N, Hkv, d]; row b uses key (seed, kind, b, epoch). */
int32_t fdllm_synth_kv_cache(uint64_t seed, int32_t kind, int32_t batch, int32_t seq_len,
                             int32_t n_kv_heads, int32_t head_dim, int64_t epoch, float sigma,
                             int32_t dtype, void *out, fdllm_stream_t stream);

/* fdllm_synth_kv_cache with the epoch taken as epoch + *epoch_add / epoch_div, epoch_add a device int64
 * read when the kernel runs (NULL: epoch alone; epoch_div >= 1): a cache refresh inside a captured CUDA
 * graph whose step counter lives on the device (refresh epoch = base + step / r). */
int32_t fdllm_synth_kv_cache_at(uint64_t seed, int32_t kind, int32_t batch, int32_t seq_len, int32_t n_kv_heads,
                                int32_t head_dim, int64_t epoch, const int64_t *epoch_add, int64_t epoch_div,
                                float sigma, int32_t dtype, void *out, fdllm_stream_t stream);

/* Per-position rows: out [b, npos, width]; row (b, p) uses key (seed, kind, b, step, pos0 + p).
 * width (and hidden below) at most 65535 * 512; FDLLM_EINVAL otherwise. */
int32_t fdllm_synth_rows(uint64_t seed, int32_t kind, int32_t batch, int64_t step, int32_t pos0,
                         int32_t npos, int32_t width, float sigma, int32_t dtype, void *out,
                         fdllm_stream_t stream);

/* Hidden-state rows out [b, npos, H]: z + 6 * W[t] (float32 multiply then add,
 * each rounded to nearest even) where the (b, step, pos) plant draw is below
 * p_plant, else z; `w` is the stored LM-head weight [V, H] in `dtype`. */
int32_t fdllm_synth_hidden(uint64_t seed, int32_t batch, int64_t step, int32_t pos0, int32_t npos,
                           int32_t hidden, int32_t vocab, double p_plant, const void *w,
                           int32_t dtype, void *out, fdllm_stream_t stream);

/* fdllm_synth_rows / fdllm_synth_hidden with the step taken as step + *step_add, step_add a device
 * int64 read when the kernel runs (NULL: step alone): per-step inputs inside a captured CUDA graph
 * whose step counter lives on the device. */
int32_t fdllm_synth_rows_at(uint64_t seed, int32_t kind, int32_t batch, int64_t step, const int64_t *step_add,
                            int32_t pos0, int32_t npos, int32_t width, float sigma, int32_t dtype, void *out,
                            fdllm_stream_t stream);
int32_t fdllm_synth_hidden_at(uint64_t seed, int32_t batch, int64_t step, const int64_t *step_add, int32_t pos0,
                              int32_t npos, int32_t hidden, int32_t vocab, double p_plant, const void *w,
                              int32_t dtype, void *out, fdllm_stream_t stream);

/* Per-sequence forms, for sequences that each sit at their own block and step (a generation in which
 * every sequence moves to its next block on its own): sequence b uses step[b] and positions
 * pos0[b] + p (device int32 [b] arrays read when the kernel runs), the same keys as the lock-step calls
 * above with that step and position. */
int32_t fdllm_synth_rows_seq(uint64_t seed, int32_t kind, int32_t batch, const int32_t *step, const int32_t *pos0,
                             int32_t npos, int32_t width, float sigma, int32_t dtype, void *out,
                             fdllm_stream_t stream);
int32_t fdllm_synth_hidden_seq(uint64_t seed, int32_t batch, const int32_t *step, const int32_t *pos0, int32_t npos,
                               int32_t hidden, int32_t vocab, double p_plant, const void *w, int32_t dtype, void *out,
                               fdllm_stream_t stream);
/* Cache rows of sequence b drawn for refresh epoch epoch[b] (device int32 [b]) into out [b, N, Hkv, d], only
 * for the sequences whose only[b] is nonzero (device uint8 [b]; NULL: every sequence); the others are left
 * untouched. */
int32_t fdllm_synth_kv_cache_seq(uint64_t seed, int32_t kind, int32_t batch, int32_t seq_len, int32_t n_kv_heads,
                                 int32_t head_dim, const int32_t *epoch, const uint8_t *only, float sigma,
                                 int32_t dtype, void *out, fdllm_stream_t stream);

/* Prompt ids out int32 [b, P], uniform over [0, vocab). */
int32_t fdllm_synth_prompt(uint64_t seed, int32_t batch, int32_t prompt_len, int32_t vocab,
                           int32_t *out, fdllm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FDLLM_SYNTH_H_ */
