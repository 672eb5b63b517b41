// Device twin of the seeded synthetic input generator (see include/fdllm_synth.h).
// Integer SplitMix64 + Irwin-Hall-12 normals, explicit round-to-nearest float32
// operations (no FMA contraction) and round-to-nearest-even bf16 stores, so the
// bytes equal the host generator's.
#include "../../include/fdllm_synth.h"
#include "common.cuh"
#include "internal.h"

namespace fdllm {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t fmix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__host__ __device__ __forceinline__ uint64_t splitmix(uint64_t state, uint64_t i) {
  return fmix(state + (i + 1) * kGamma);
}

__device__ __forceinline__ float normal12(uint64_t key, uint64_t idx) {
  int64_t tot = 0;
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const uint64_t r = splitmix(key, idx * 3 + part);
    tot += (int64_t)(r & 0xFFFF) + (int64_t)((r >> 16) & 0xFFFF) + (int64_t)((r >> 32) & 0xFFFF) +
           (int64_t)(r >> 48);
  }
  return __fdiv_rn((float)(tot - 393210), 65536.0f);  // exact: integer over a power of two
}

template <typename T> __device__ __forceinline__ void store(T *p, float v);
template <> __device__ __forceinline__ void store<float>(float *p, float v) { *p = v; }
template <> __device__ __forceinline__ void store<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename T>
__global__ void normals_kernel(uint64_t key, int64_t n, int64_t offset, float sigma, T *out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    store(out + i, __fmul_rn(normal12(key, (uint64_t)(offset + i)), sigma));
}

// one stream per (b, epoch): out [b, per]; per-sequence epochs and a sequence filter when given
template <typename T>
__global__ void kv_kernel(uint64_t seed, int kind, int64_t epoch, int64_t per, float sigma, T *out,
                          const int64_t *epoch_add = nullptr, int64_t epoch_div = 1,
                          const int32_t *epoch_seq = nullptr, const uint8_t *only = nullptr) {
  const int b = blockIdx.y;
  if (only != nullptr && only[b] == 0) return;
  if (epoch_seq != nullptr) epoch = epoch_seq[b];
  if (epoch_add != nullptr) epoch += *epoch_add / epoch_div;
  const uint64_t key = splitmix(splitmix(splitmix(seed, (uint64_t)kind), (uint64_t)b), (uint64_t)epoch);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per;
       i += (int64_t)gridDim.x * blockDim.x)
    store(out + (int64_t)b * per + i, __fmul_rn(normal12(key, (uint64_t)i), sigma));
}

__device__ __forceinline__ uint64_t row_key(uint64_t seed, int kind, int b, int64_t step, int64_t pos) {
  return splitmix(splitmix(splitmix(splitmix(seed, (uint64_t)kind), (uint64_t)b), (uint64_t)step),
                  (uint64_t)pos);
}

constexpr int kRowChunk = 512;   // row elements per CTA (grid z): short row batches still fill the GPU

// rows [b, npos, width]: grid (npos, b, row chunks); the step is step + *step_add when step_add is given (a device
// counter, e.g. a graph loop's); per-sequence steps and first positions when step_seq / pos_seq are given
template <typename T>
__global__ void rows_kernel(uint64_t seed, int kind, int64_t step, const int64_t *step_add, int pos0, int npos,
                            int width, float sigma, T *out, const int32_t *step_seq = nullptr,
                            const int32_t *pos_seq = nullptr) {
  const int p = blockIdx.x, b = blockIdx.y;
  if (step_add != nullptr) step += *step_add;
  if (step_seq != nullptr) step = step_seq[b];
  if (pos_seq != nullptr) pos0 = pos_seq[b];
  const uint64_t key = row_key(seed, kind, b, step, pos0 + p);
  T *row = out + ((int64_t)b * npos + p) * width;
  const int i1 = min(width, ((int)blockIdx.z + 1) * kRowChunk);
  for (int i = (int)blockIdx.z * kRowChunk + threadIdx.x; i < i1; i += blockDim.x)
    store(row + i, __fmul_rn(normal12(key, (uint64_t)i), sigma));
}

template <typename T>
__global__ void hidden_kernel(uint64_t seed, int64_t step, const int64_t *step_add, int pos0, int npos, int hidden,
                              int vocab, uint64_t plant_thr, const T *w, T *out, const int32_t *step_seq = nullptr,
                              const int32_t *pos_seq = nullptr) {
  const int p = blockIdx.x, b = blockIdx.y;
  if (step_add != nullptr) step += *step_add;
  if (step_seq != nullptr) step = step_seq[b];
  if (pos_seq != nullptr) pos0 = pos_seq[b];
  const uint64_t pk = row_key(seed, FDLLM_SYNTH_PLANT, b, step, pos0 + p);
  const bool planted = (splitmix(pk, 0) >> 40) < plant_thr;
  const int64_t target = (int64_t)(((splitmix(pk, 1) >> 32) * (uint64_t)vocab) >> 32);
  const uint64_t key = row_key(seed, FDLLM_SYNTH_HID, b, step, pos0 + p);
  T *row = out + ((int64_t)b * npos + p) * hidden;
  const int i1 = min(hidden, ((int)blockIdx.z + 1) * kRowChunk);
  for (int i = (int)blockIdx.z * kRowChunk + threadIdx.x; i < i1; i += blockDim.x) {
    float z = normal12(key, (uint64_t)i);
    if (planted) z = __fadd_rn(z, __fmul_rn(6.0f, to_f32(w[target * hidden + i])));
    store(row + i, z);
  }
}

__global__ void prompt_kernel(uint64_t seed, int prompt_len, int vocab, int32_t *out) {
  const int b = blockIdx.y;
  const uint64_t key = splitmix(splitmix(seed, (uint64_t)FDLLM_SYNTH_PROMPT), (uint64_t)b);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < prompt_len; i += gridDim.x * blockDim.x)
    out[(int64_t)b * prompt_len + i] = (int32_t)(((splitmix(key, (uint64_t)i) >> 32) * (uint64_t)vocab) >> 32);
}

int32_t finish() { return cudaGetLastError() == cudaSuccess ? FDLLM_OK : FDLLM_ECUDA; }

unsigned grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 16;
  return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace
}  // namespace fdllm

using namespace fdllm;

extern "C" int32_t fdllm_synth_normals(uint64_t seed, int32_t kind, const int64_t *coords,
                                       int32_t n_coords, int64_t n, int64_t offset, float sigma,
                                       int32_t dtype, void *out, fdllm_stream_t stream) {
  if (n < 0 || offset < 0 || n_coords < 0 || n_coords > 4 || (n_coords > 0 && !coords) ||
      (n > 0 && !out) || (dtype != FDLLM_BF16 && dtype != FDLLM_F32))
    return FDLLM_EINVAL;
  if (n == 0) return FDLLM_OK;
  uint64_t key = splitmix(seed, (uint64_t)kind);
  for (int i = 0; i < n_coords; ++i) key = splitmix(key, (uint64_t)coords[i]);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    normals_kernel<<<grid_for(n), 256, 0, st>>>(key, n, offset, sigma, (__nv_bfloat16 *)out);
  else
    normals_kernel<<<grid_for(n), 256, 0, st>>>(key, n, offset, sigma, (float *)out);
  return finish();
}

extern "C" int32_t fdllm_synth_kv_cache(uint64_t seed, int32_t kind, int32_t batch, int32_t seq_len,
                                        int32_t n_kv_heads, int32_t head_dim, int64_t epoch,
                                        float sigma, int32_t dtype, void *out,
                                        fdllm_stream_t stream) {
  return fdllm_synth_kv_cache_at(seed, kind, batch, seq_len, n_kv_heads, head_dim, epoch, nullptr, 1, sigma, dtype,
                                 out, stream);
}

extern "C" int32_t fdllm_synth_kv_cache_at(uint64_t seed, int32_t kind, int32_t batch, int32_t seq_len,
                                           int32_t n_kv_heads, int32_t head_dim, int64_t epoch,
                                           const int64_t *epoch_add, int64_t epoch_div, float sigma, int32_t dtype,
                                           void *out, fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || seq_len < 1 || n_kv_heads < 1 || head_dim < 1 || !out || epoch_div < 1 ||
      (dtype != FDLLM_BF16 && dtype != FDLLM_F32))
    return FDLLM_EINVAL;
  const int64_t per = (int64_t)seq_len * n_kv_heads * head_dim;
  dim3 grid(grid_for(per) / (unsigned)batch + 1, batch);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    kv_kernel<<<grid, 256, 0, st>>>(seed, kind, epoch, per, sigma, (__nv_bfloat16 *)out, epoch_add, epoch_div);
  else
    kv_kernel<<<grid, 256, 0, st>>>(seed, kind, epoch, per, sigma, (float *)out, epoch_add, epoch_div);
  return finish();
}

extern "C" int32_t fdllm_synth_rows(uint64_t seed, int32_t kind, int32_t batch, int64_t step,
                                    int32_t pos0, int32_t npos, int32_t width, float sigma,
                                    int32_t dtype, void *out, fdllm_stream_t stream) {
  return fdllm_synth_rows_at(seed, kind, batch, step, nullptr, pos0, npos, width, sigma, dtype, out, stream);
}

extern "C" int32_t fdllm_synth_rows_at(uint64_t seed, int32_t kind, int32_t batch, int64_t step,
                                       const int64_t *step_add, int32_t pos0, int32_t npos, int32_t width,
                                       float sigma, int32_t dtype, void *out, fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || npos < 0 || width < 1 || width > 65535 * kRowChunk || (npos > 0 && !out) ||
      (dtype != FDLLM_BF16 && dtype != FDLLM_F32))
    return FDLLM_EINVAL;
  if (npos == 0) return FDLLM_OK;
  dim3 grid(npos, batch, (width + kRowChunk - 1) / kRowChunk);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    rows_kernel<<<grid, 128, 0, st>>>(seed, kind, step, step_add, pos0, npos, width, sigma, (__nv_bfloat16 *)out);
  else
    rows_kernel<<<grid, 128, 0, st>>>(seed, kind, step, step_add, pos0, npos, width, sigma, (float *)out);
  return finish();
}

extern "C" int32_t fdllm_synth_hidden(uint64_t seed, int32_t batch, int64_t step, int32_t pos0,
                                      int32_t npos, int32_t hidden, int32_t vocab, double p_plant,
                                      const void *w, int32_t dtype, void *out,
                                      fdllm_stream_t stream) {
  return fdllm_synth_hidden_at(seed, batch, step, nullptr, pos0, npos, hidden, vocab, p_plant, w, dtype, out, stream);
}

extern "C" int32_t fdllm_synth_hidden_at(uint64_t seed, int32_t batch, int64_t step, const int64_t *step_add,
                                         int32_t pos0, int32_t npos, int32_t hidden, int32_t vocab, double p_plant,
                                         const void *w, int32_t dtype, void *out, fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || npos < 0 || hidden < 1 || hidden > 65535 * kRowChunk || vocab < 1 || !w ||
      (npos > 0 && !out) || (dtype != FDLLM_BF16 && dtype != FDLLM_F32) || !(p_plant >= 0.0))
    return FDLLM_EINVAL;
  if (npos == 0) return FDLLM_OK;
  // plant iff (draw >> 40) < floor(p * 2^24), as on the host
  const uint64_t thr = (uint64_t)floor(p_plant * (double)(1 << 24));
  dim3 grid(npos, batch, (hidden + kRowChunk - 1) / kRowChunk);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    hidden_kernel<<<grid, 128, 0, st>>>(seed, step, step_add, pos0, npos, hidden, vocab, thr,
                                        (const __nv_bfloat16 *)w, (__nv_bfloat16 *)out);
  else
    hidden_kernel<<<grid, 128, 0, st>>>(seed, step, step_add, pos0, npos, hidden, vocab, thr, (const float *)w,
                                        (float *)out);
  return finish();
}

extern "C" int32_t fdllm_synth_rows_seq(uint64_t seed, int32_t kind, int32_t batch, const int32_t *step,
                                        const int32_t *pos0, int32_t npos, int32_t width, float sigma, int32_t dtype,
                                        void *out, fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || npos < 0 || width < 1 || width > 65535 * kRowChunk || !step || !pos0 ||
      (npos > 0 && !out) ||
      (dtype != FDLLM_BF16 && dtype != FDLLM_F32))
    return FDLLM_EINVAL;
  if (npos == 0) return FDLLM_OK;
  dim3 grid(npos, batch, (width + kRowChunk - 1) / kRowChunk);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    rows_kernel<<<grid, 128, 0, st>>>(seed, kind, 0, nullptr, 0, npos, width, sigma, (__nv_bfloat16 *)out, step,
                                      pos0);
  else
    rows_kernel<<<grid, 128, 0, st>>>(seed, kind, 0, nullptr, 0, npos, width, sigma, (float *)out, step, pos0);
  return finish();
}

extern "C" int32_t fdllm_synth_hidden_seq(uint64_t seed, int32_t batch, const int32_t *step, const int32_t *pos0,
                                          int32_t npos, int32_t hidden, int32_t vocab, double p_plant, const void *w,
                                          int32_t dtype, void *out, fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || npos < 0 || hidden < 1 || hidden > 65535 * kRowChunk || vocab < 1 || !w ||
      !step || !pos0 ||
      (npos > 0 && !out) || (dtype != FDLLM_BF16 && dtype != FDLLM_F32) || !(p_plant >= 0.0))
    return FDLLM_EINVAL;
  if (npos == 0) return FDLLM_OK;
  const uint64_t thr = (uint64_t)floor(p_plant * (double)(1 << 24));
  dim3 grid(npos, batch, (hidden + kRowChunk - 1) / kRowChunk);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    hidden_kernel<<<grid, 128, 0, st>>>(seed, 0, nullptr, 0, npos, hidden, vocab, thr, (const __nv_bfloat16 *)w,
                                        (__nv_bfloat16 *)out, step, pos0);
  else
    hidden_kernel<<<grid, 128, 0, st>>>(seed, 0, nullptr, 0, npos, hidden, vocab, thr, (const float *)w,
                                        (float *)out, step, pos0);
  return finish();
}

extern "C" int32_t fdllm_synth_kv_cache_seq(uint64_t seed, int32_t kind, int32_t batch, int32_t seq_len,
                                            int32_t n_kv_heads, int32_t head_dim, const int32_t *epoch,
                                            const uint8_t *only, float sigma, int32_t dtype, void *out,
                                            fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || seq_len < 1 || n_kv_heads < 1 || head_dim < 1 || !out || !epoch ||
      (dtype != FDLLM_BF16 && dtype != FDLLM_F32))
    return FDLLM_EINVAL;
  const int64_t per = (int64_t)seq_len * n_kv_heads * head_dim;
  dim3 grid(grid_for(per) / (unsigned)batch + 1, batch);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == FDLLM_BF16)
    kv_kernel<<<grid, 256, 0, st>>>(seed, kind, 0, per, sigma, (__nv_bfloat16 *)out, nullptr, 1, epoch, only);
  else
    kv_kernel<<<grid, 256, 0, st>>>(seed, kind, 0, per, sigma, (float *)out, nullptr, 1, epoch, only);
  return finish();
}

extern "C" int32_t fdllm_synth_prompt(uint64_t seed, int32_t batch, int32_t prompt_len,
                                      int32_t vocab, int32_t *out, fdllm_stream_t stream) {
  if (batch < 1 || batch > 65535 || prompt_len < 0 || vocab < 1 || (prompt_len > 0 && !out))
    return FDLLM_EINVAL;
  if (prompt_len == 0) return FDLLM_OK;
  dim3 grid((prompt_len + 255) / 256, batch);
  prompt_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(seed, prompt_len, vocab, out);
  return finish();
}
