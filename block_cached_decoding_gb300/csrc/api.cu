// Host side of the C ABI declared in include/fdllm.h: argument validation,
// workspace layout, dispatch to the kernels, status codes and error messages.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {

// Per-device error word for bounded device waits (see fdllm_last_device_error).
__device__ int32_t g_device_error_word = 0;

namespace {

thread_local std::string t_last_error;

// One thread waits on an mbarrier that expects an arrival nobody makes.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  tc::fence_barrier_init();
  if (!tc::mbar_wait(&bar, 0, limit_ns)) record_device_error(err, 900);
}

fdllm_status fail(fdllm_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

fdllm_status cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return FDLLM_OK;
  return fail(FDLLM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The clustered LM head multicasts tiles of its operands between the CTAs of a cluster; it is
// meant for memory of this GPU only, so each operand must be device memory (cudaMalloc, torch)
// of the current device: host, managed or another device's memory is rejected.
fdllm_status check_local_device(const void *ptr, const char *what) {
  int dev = 0;
  fdllm_status st = cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != FDLLM_OK) return st;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(FDLLM_EINVAL, "select: %s is not CUDA device memory", what);
  }
  if (at.type != cudaMemoryTypeDevice || at.device != dev)
    return fail(FDLLM_EINVAL,
                "select: with more than 128 block rows, %s must be device memory of the current device "
                "(memory type %d on device %d; current device %d)",
                what, (int)at.type, at.device, dev);
  return FDLLM_OK;
}

// The LM head's operands (hidden rows or their E4M3 copy, weight) when the clustered kernel runs.
fdllm_status check_cluster_operands(const SelectProblem &p, bool tc, const void *hidden, const void *w) {
  if (!tc || !lmhead_tc_clustered(p)) return FDLLM_OK;
  fdllm_status st = check_local_device(hidden, "hidden");
  if (st != FDLLM_OK) return st;
  return check_local_device(w, "lm_head_w");
}

constexpr int kMaxDevices = 64;

// The calling thread's current CUDA context, or null if it cannot be read.  A device address of a
// __device__ variable is valid only in the context it was looked up in (a device reset creates a
// new primary context), so cached addresses are keyed by it.
void *current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return (PFN_cuCtxGetCurrent_v4000)p;
    return (PFN_cuCtxGetCurrent_v4000) nullptr;
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return (void *)c;
}

// Device address of a __device__ symbol on the current device, looked up with
// cudaGetSymbolAddress the first time it is needed in each (device, context) and cached.
struct SymbolCache {
  std::mutex mu;
  void *ctx[kMaxDevices] = {nullptr};
  void *ptr[kMaxDevices] = {nullptr};

  cudaError_t get(const void *symbol, void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // make sure the device's primary context exists (the lookup below would create it too)
    void *c = current_context();
    std::lock_guard<std::mutex> lk(mu);
    if (!ptr[dev] || c == nullptr || ctx[dev] != c) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, symbol);
      if (e != cudaSuccess) return e;
      ptr[dev] = p;
      ctx[dev] = current_context();
    }
    *out = ptr[dev];
    return cudaSuccess;
  }
};

int32_t *error_word_ptr() {
  static SymbolCache cache;
  void *p = nullptr;
  return cache.get((const void *)&g_device_error_word, &p) == cudaSuccess ? (int32_t *)p : nullptr;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------------------
// attention
// ----------------------------------------------------------------------------
fdllm_status resolve_attn(const fdllm_attn_desc *d, AttnProblem &p) {
  if (!d) return fail(FDLLM_EINVAL, "attn: null descriptor");
  if (d->batch < 1) return fail(FDLLM_EINVAL, "attn: batch must be >= 1 (got %d)", d->batch);
  if (d->prompt_len < 0) return fail(FDLLM_EINVAL, "attn: prompt_len < 0");
  if (d->block_size < 1) return fail(FDLLM_EINVAL, "attn: block_size must be >= 1");
  if (d->gen_length < d->block_size || d->gen_length % d->block_size != 0)
    return fail(FDLLM_EINVAL, "attn: gen_length (%d) must be a positive multiple of block_size (%d)",
                d->gen_length, d->block_size);
  const int nblocks = d->gen_length / d->block_size;
  if (d->block_idx < 0 || d->block_idx >= nblocks)
    return fail(FDLLM_EINVAL, "attn: block_idx %d outside [0, %d)", d->block_idx, nblocks);
  if (d->n_kv_heads < 1 || d->n_q_heads < 1 || d->n_q_heads % d->n_kv_heads != 0)
    return fail(FDLLM_EINVAL, "attn: n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                d->n_q_heads, d->n_kv_heads);
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(FDLLM_EINVAL, "attn: head_dim must be 64 or 128 (got %d)", d->head_dim);
  if (d->use_cache != 0 && d->use_cache != 1) return fail(FDLLM_EINVAL, "attn: use_cache must be 0 or 1");
  if (d->dual_cache != 0 && d->dual_cache != 1) return fail(FDLLM_EINVAL, "attn: dual_cache must be 0 or 1");
  if (d->dtype != FDLLM_BF16 && d->dtype != FDLLM_F32) return fail(FDLLM_EINVAL, "attn: bad dtype %d", d->dtype);
  if (d->out_f32 != 0 && d->out_f32 != 1) return fail(FDLLM_EINVAL, "attn: out_f32 must be 0 or 1");
  if (!(d->sm_scale >= 0.f) || isinf(d->sm_scale)) return fail(FDLLM_EINVAL, "attn: sm_scale must be finite and >= 0");
  const int64_t n = (int64_t)d->prompt_len + d->gen_length;
  if (n > (1 << 24)) return fail(FDLLM_EINVAL, "attn: sequence too long");
  const int s = d->prompt_len + d->block_idx * d->block_size;
  p.batch = d->batch;
  p.seq_len = (int)n;
  p.blocks = nullptr;
  p.prompt_len = d->prompt_len;
  p.nblocks = nblocks;
  p.hq = d->n_q_heads;
  p.hkv = d->n_kv_heads;
  p.d = d->head_dim;
  if (!d->use_cache) {
    p.fresh0 = 0;
    p.nq = (int)n;
  } else if (d->dual_cache) {
    p.fresh0 = s;
    p.nq = d->block_size;
  } else {
    p.fresh0 = s;
    p.nq = (int)n - s;
  }
  p.scale = d->sm_scale > 0.f ? d->sm_scale : (float)(1.0 / sqrt((double)d->head_dim));
  p.in_bf16 = d->dtype == FDLLM_BF16;
  p.out_f32 = d->out_f32;
  p.f8kv = 0;
  p.k_scale = p.v_scale = nullptr;
  p.update = 0;
  p.win = d->block_size;
  p.kc_w = p.vc_w = nullptr;
  return FDLLM_OK;
}

}  // namespace

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int sm_count() {
  static int counts[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  if (!counts[dev]) {
    int c = 0;
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = c > 0 ? c : 1;
  }
  return counts[dev];
}

namespace {

// ----------------------------------------------------------------------------
// select
// ----------------------------------------------------------------------------
fdllm_status resolve_select(const fdllm_select_desc *d, SelectProblem &p) {
  if (!d) return fail(FDLLM_EINVAL, "select: null descriptor");
  if (d->batch < 1) return fail(FDLLM_EINVAL, "select: batch must be >= 1");
  if (d->block_size < 1 || d->block_size > 256)
    return fail(FDLLM_EINVAL, "select: block_size must be in [1, 256] (got %d)", d->block_size);
  if (d->block_start < 0 || d->seq_len < 1 || (int64_t)d->block_start + d->block_size > d->seq_len)
    return fail(FDLLM_EINVAL, "select: block [%d, %d) outside the sequence of length %d", d->block_start,
                d->block_start + d->block_size, d->seq_len);
  if (d->hidden < 64 || d->hidden % 64 != 0)
    return fail(FDLLM_EINVAL, "select: hidden must be a positive multiple of 64 (got %d)", d->hidden);
  if (d->vocab < 2) return fail(FDLLM_EINVAL, "select: vocab must be >= 2");
  if ((int64_t)d->batch * d->block_size > 2048)
    return fail(FDLLM_EINVAL, "select: batch * block_size must be <= 2048");
  if (d->mask_id >= 0 && d->mask_id < d->vocab)
    return fail(FDLLM_EINVAL, "select: mask_id %d is a vocabulary id; it must lie outside [0, vocab)", d->mask_id);
  if (d->dtype != FDLLM_BF16 && d->dtype != FDLLM_F32) return fail(FDLLM_EINVAL, "select: bad dtype %d", d->dtype);
  switch (d->strategy) {
    case FDLLM_SELECT_THRESHOLD:
      if (isnan(d->threshold)) return fail(FDLLM_EINVAL, "select: threshold is NaN");
      break;
    case FDLLM_SELECT_FACTOR:
      if (!(d->factor > 0.f)) return fail(FDLLM_EINVAL, "select: factor must be > 0");
      break;
    case FDLLM_SELECT_TOPK:
      if (d->topk < 1) return fail(FDLLM_EINVAL, "select: topk must be >= 1");
      break;
    default:
      return fail(FDLLM_EINVAL, "select: unknown strategy %d", d->strategy);
  }
  p.batch = d->batch;
  p.seq_len = d->seq_len;
  p.s = d->block_start;
  p.starts = nullptr;
  p.B = d->block_size;
  p.H = d->hidden;
  p.V = d->vocab;
  p.mask_id = d->mask_id;
  p.strategy = d->strategy;
  p.topk = d->topk;
  p.factor = d->factor;
  const double tau = d->threshold;
  // c > tau  <=>  log((1 - c) / c) < log((1 - tau) / tau)
  p.kappa_tau = tau >= 1.0 ? -INFINITY : (tau <= 0.0 ? INFINITY : (float)log((1.0 - tau) / tau));
  p.in_bf16 = d->dtype == FDLLM_BF16;
  p.fp8w = 0;
  p.quant_hidden = 0;
  p.w_scale = nullptr;
  p.h_scale = nullptr;
  p.hq = nullptr;
  return FDLLM_OK;
}

// workspace: [8-byte tickets: arrivals, starts, selectors done, quantised rows] [partials
// VocabStat [b * B, splits], 16 bytes each, from byte 256]; the tensor-core kernel serves bf16
// blocks of up to 512 rows (and runs the select itself), the CUDA-core kernel the
// rest (followed by select_kernel)
struct SelectLayout {
  size_t part_off, total;
  size_t hq_off, hs_off;   // FP8 weight cache: the quantised hidden rows and their scales
  int splits;
  bool tc;
};

SelectLayout select_layout(const SelectProblem &p) {
  SelectLayout L;
  L.tc = lmhead_tc_supported(p);
  L.splits = L.tc ? lmhead_tc_grid(p) : lmhead_simt_splits(p);
  // the tickets, then the partials
  L.part_off = 256;
  L.total = L.part_off + align_up((size_t)p.batch * p.B * L.splits * sizeof(VocabStat), 256);
  L.hq_off = L.hs_off = 0;
  if (p.fp8w) {
    const size_t rows = (size_t)p.batch * p.B;
    L.hq_off = L.total;
    L.hs_off = L.hq_off + align_up(rows * p.H, 256);
    L.total = L.hs_off + align_up(rows * sizeof(float), 256);
  }
  return L;
}

// LM head + select on the partials at `ws` (laid out by select_layout)
cudaError_t run_select(const SelectProblem &p, const SelectLayout &L, void *ws, cudaStream_t st) {
  VocabStat *part = (VocabStat *)((char *)ws + L.part_off);
  if (p.fp8w) {
    // the block's hidden rows in E4M3 (per-row scales), then the E4M3 LM head
    SelectProblem q = p;
    q.hq = (char *)ws + L.hq_off;
    q.h_scale = (const float *)((char *)ws + L.hs_off);
    q.quant_hidden = lmhead_tc_quantises_hidden(p) ? 1 : 0;   // else the row quantiser runs first
    if (!q.quant_hidden) {
      cudaError_t e = launch_quantize_fp8(p.hidden, true, (int64_t)p.batch * p.B, p.H, (uint8_t *)q.hq,
                                          (float *)q.h_scale, st);
      if (e != cudaSuccess) return e;
    }
    return launch_lmhead_tc(q, part, (unsigned long long *)ws, L.splits, st);
  }
  if (L.tc) return launch_lmhead_tc(p, part, (unsigned long long *)ws, L.splits, st);
  cudaError_t e = launch_lmhead_simt(p, part, L.splits, st);
  if (e != cudaSuccess) return e;
  return launch_select(p, part, L.splits, st);
}

}  // namespace
}  // namespace fdllm

using namespace fdllm;

extern "C" {

int32_t fdllm_version(void) { return 106; }

fdllm_status fdllm_selftest_bounded_wait(int32_t limit_ms, fdllm_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 1000) return fail(FDLLM_EINVAL, "selftest: limit_ms must be in 1..1000");
  int32_t *err = error_word_ptr();
  if (!err) return fail(FDLLM_ECUDA, "selftest: device error word unavailable");
  selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ms * 1000000ull, err);
  count_launches(1);
  return cuda_status(cudaGetLastError(), "selftest launch");
}

uint64_t fdllm_launch_counter(void) { return g_launches.load(std::memory_order_relaxed); }

const char *fdllm_status_string(int32_t s) {
  switch (s) {
    case FDLLM_OK: return "FDLLM_OK: success";
    case FDLLM_EINVAL: return "FDLLM_EINVAL: invalid argument";
    case FDLLM_ECUDA: return "FDLLM_ECUDA: CUDA runtime error";
    case FDLLM_ETIMEOUT: return "FDLLM_ETIMEOUT: a bounded device wait expired";
    case FDLLM_EUNSUPPORTED: return "FDLLM_EUNSUPPORTED: not supported by this build";
    default: return "unknown fdllm status";
  }
}

const char *fdllm_last_error(void) { return t_last_error.c_str(); }

fdllm_status fdllm_last_device_error(fdllm_stream_t stream, int32_t *detail) {
  fdllm_status st = cuda_status(cudaStreamSynchronize((cudaStream_t)stream), "stream synchronize");
  if (st != FDLLM_OK) return st;
  int32_t *w = error_word_ptr();
  if (!w) return fail(FDLLM_ECUDA, "device error word unavailable");
  int32_t v = 0;
  st = cuda_status(cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost), "read device error word");
  if (st != FDLLM_OK) return st;
  if (v != 0) {
    const int32_t zero = 0;
    st = cuda_status(cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice), "clear device error word");
    if (st != FDLLM_OK) return st;
  }
  if (detail) *detail = v;
  if (v >= 231 && v <= 233) return fail(FDLLM_EINVAL, "per-sequence block index out of range (site %d)", v);
  return v ? fail(FDLLM_ETIMEOUT, "device wait gave up at site %d", v) : FDLLM_OK;
}

int64_t fdllm_attn_query_count(const fdllm_attn_desc *desc) {
  AttnProblem p;
  if (resolve_attn(desc, p) != FDLLM_OK) return -1;
  return p.nq;
}

static size_t attn_workspace(const AttnProblem &p) {
  return attn_tc_supported(p) ? attn_tc_workspace(p) : attn_simt_workspace(p);
}

size_t fdllm_attn_workspace_size(const fdllm_attn_desc *desc) {
  AttnProblem p;
  if (resolve_attn(desc, p) != FDLLM_OK) return 0;
  return attn_workspace(p);
}

// k_scale / v_scale non-null: the caches are E4M3 codes with per-row scales (the FP8 KV cache)
static fdllm_status block_attn(const fdllm_attn_desc *desc, const int32_t *blocks, const void *q,
                               const void *k_cache, const void *v_cache, const void *k_fresh,
                               const void *v_fresh, void *out, float *lse, void *workspace, size_t ws_bytes,
                               fdllm_stream_t stream, const float *k_scale = nullptr,
                               const float *v_scale = nullptr, bool update = false) {
  AttnProblem p;
  fdllm_status st = resolve_attn(desc, p);
  if (st != FDLLM_OK) return st;
  if (update) {
    if (!desc->use_cache)
      return fail(FDLLM_EUNSUPPORTED, "attn update: the window update needs a cache (use_cache = 1)");
    p.update = 1;
    p.kc_w = const_cast<void *>(k_cache);
    p.vc_w = const_cast<void *>(v_cache);
  }
  if (k_scale || v_scale) {
    if (!k_scale || !v_scale) return fail(FDLLM_EINVAL, "attn fp8kv: k_scale and v_scale are required");
    if (!desc->use_cache || !attn_tc_supported(p))
      return fail(FDLLM_EUNSUPPORTED, "attn fp8kv: needs a cache (use_cache = 1) and bf16 queries and fresh K/V");
    p.f8kv = 1;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
  }
  if (blocks) {
    if (!desc->use_cache || !desc->dual_cache || !attn_tc_supported(p))
      return fail(FDLLM_EUNSUPPORTED, "attn: per-sequence blocks need DualCache and bf16");
    p.blocks = blocks;
  }
  const void *req[] = {q, k_cache, v_cache, k_fresh, v_fresh, out};
  const char *names[] = {"q", "k_cache", "v_cache", "k_fresh", "v_fresh", "out"};
  for (int i = 0; i < 6; ++i) {
    if (!req[i]) return fail(FDLLM_EINVAL, "attn: %s is null", names[i]);
    if (!aligned16(req[i])) return fail(FDLLM_EINVAL, "attn: %s is not 16-byte aligned", names[i]);
  }
  const size_t need = attn_workspace(p);
  if (ws_bytes < need || (need && !workspace))
    return fail(FDLLM_EINVAL, "attn: workspace of %zu bytes is smaller than the %zu required", ws_bytes, need);
  p.q = q; p.kc = k_cache; p.vc = v_cache; p.kf = k_fresh; p.vf = v_fresh;
  if (workspace && !aligned16(workspace)) return fail(FDLLM_EINVAL, "attn: workspace must be 16-byte aligned");
  p.out = out; p.lse = lse; p.ws = workspace; p.ws_bytes = ws_bytes;
  p.err = error_word_ptr();
  cudaStream_t cs = (cudaStream_t)stream;
  if (p.update && !attn_tc_fuses_update(p)) {
    // the kernel cannot store this window itself: the attention, then the splice kernel (the block's
    // fresh rows are the whole fresh tensor only under DualCache)
    if (blocks || !desc->dual_cache)
      return fail(FDLLM_EUNSUPPORTED,
                  "attn update: the window (block_size %d) must fill whole key tiles for per-sequence blocks or "
                  "PrefixCache", desc->block_size);
    p.update = 0;
    st = cuda_status(attn_tc_supported(p) ? launch_attn_tc(p, cs) : launch_attn_simt(p, cs), "attn launch");
    if (st != FDLLM_OK) return st;
    const int64_t row_bytes = (int64_t)p.hkv * p.d * (p.in_bf16 ? 2 : 4);
    return cuda_status(launch_splice(p.batch, p.seq_len, row_bytes, p.fresh0, p.win, p.kc_w, p.vc_w, k_fresh,
                                     v_fresh, cs),
                       "attn update: splice launch");
  }
  return cuda_status(attn_tc_supported(p) ? launch_attn_tc(p, cs) : launch_attn_simt(p, cs), "attn launch");
}

fdllm_status fdllm_block_attn(const fdllm_attn_desc *desc, const void *q, const void *k_cache,
                              const void *v_cache, const void *k_fresh, const void *v_fresh,
                              void *out, float *lse, void *workspace, size_t ws_bytes,
                              fdllm_stream_t stream) {
  return block_attn(desc, nullptr, q, k_cache, v_cache, k_fresh, v_fresh, out, lse, workspace, ws_bytes, stream);
}

fdllm_status fdllm_block_attn_ragged(const fdllm_attn_desc *desc, const int32_t *block_idx, const void *q,
                                     const void *k_cache, const void *v_cache, const void *k_fresh,
                                     const void *v_fresh, void *out, float *lse, void *workspace,
                                     size_t ws_bytes, fdllm_stream_t stream) {
  if (!block_idx) return fail(FDLLM_EINVAL, "attn: block_idx is null");
  return block_attn(desc, block_idx, q, k_cache, v_cache, k_fresh, v_fresh, out, lse, workspace, ws_bytes, stream);
}

fdllm_status fdllm_block_attn_update(const fdllm_attn_desc *desc, const int32_t *block_idx, const void *q,
                                     void *k_cache, void *v_cache, const void *k_fresh, const void *v_fresh,
                                     void *out, float *lse, void *workspace, size_t ws_bytes,
                                     fdllm_stream_t stream) {
  return block_attn(desc, block_idx, q, k_cache, v_cache, k_fresh, v_fresh, out, lse, workspace, ws_bytes, stream,
                    nullptr, nullptr, true);
}

size_t fdllm_select_workspace_size(const fdllm_select_desc *desc) {
  SelectProblem p;
  if (resolve_select(desc, p) != FDLLM_OK) return 0;
  return select_layout(p).total;
}

static fdllm_status confidence_select(const fdllm_select_desc *desc, const int32_t *starts, const void *hidden,
                                      const void *lm_head_w, int32_t *tokens, uint8_t *unmasked, float *conf,
                                      float *kappa, int32_t *argmax, int32_t *n_masked_left, void *workspace,
                                      size_t ws_bytes, fdllm_stream_t stream) {
  SelectProblem p;
  fdllm_status st = resolve_select(desc, p);
  if (st != FDLLM_OK) return st;
  p.starts = starts;
  const void *req[] = {hidden, lm_head_w, tokens, unmasked, conf, argmax, n_masked_left, workspace};
  const char *names[] = {"hidden", "lm_head_w", "tokens", "unmasked", "conf", "argmax", "n_masked_left", "workspace"};
  for (int i = 0; i < 8; ++i)
    if (!req[i]) return fail(FDLLM_EINVAL, "select: %s is null", names[i]);
  if (!aligned16(hidden) || !aligned16(lm_head_w))
    return fail(FDLLM_EINVAL, "select: hidden and lm_head_w must be 16-byte aligned");
  if (!aligned16(workspace)) return fail(FDLLM_EINVAL, "select: workspace must be 16-byte aligned");
  const SelectLayout L = select_layout(p);
  if (ws_bytes < L.total)
    return fail(FDLLM_EINVAL, "select: workspace of %zu bytes is smaller than the %zu required", ws_bytes, L.total);
  st = check_cluster_operands(p, L.tc, hidden, lm_head_w);
  if (st != FDLLM_OK) return st;
  p.hidden = hidden; p.w = lm_head_w; p.tokens = tokens; p.unmasked = unmasked; p.conf = conf;
  p.kappa = kappa; p.argmax = argmax; p.n_left = n_masked_left; p.ws = workspace; p.ws_bytes = ws_bytes;
  p.err = error_word_ptr();
  return cuda_status(run_select(p, L, workspace, (cudaStream_t)stream), "lm-head / select launch");
}

fdllm_status fdllm_confidence_select(const fdllm_select_desc *desc, const void *hidden,
                                     const void *lm_head_w, int32_t *tokens, uint8_t *unmasked,
                                     float *conf, float *kappa, int32_t *argmax,
                                     int32_t *n_masked_left, void *workspace, size_t ws_bytes,
                                     fdllm_stream_t stream) {
  return confidence_select(desc, nullptr, hidden, lm_head_w, tokens, unmasked, conf, kappa, argmax, n_masked_left,
                           workspace, ws_bytes, stream);
}

fdllm_status fdllm_confidence_select_ragged(const fdllm_select_desc *desc, const int32_t *block_start,
                                            const void *hidden, const void *lm_head_w, int32_t *tokens,
                                            uint8_t *unmasked, float *conf, float *kappa, int32_t *argmax,
                                            int32_t *n_masked_left, void *workspace, size_t ws_bytes,
                                            fdllm_stream_t stream) {
  if (!block_start) return fail(FDLLM_EINVAL, "select: block_start is null");
  return confidence_select(desc, block_start, hidden, lm_head_w, tokens, unmasked, conf, kappa, argmax,
                           n_masked_left, workspace, ws_bytes, stream);
}

// ---- FP8 weight cache ----
fdllm_status fdllm_quantize_fp8_rows(int64_t rows, int32_t cols, int32_t dtype, const void *src, uint8_t *q,
                                     float *scale, fdllm_stream_t stream) {
  if (rows < 0 || cols < 0) return fail(FDLLM_EINVAL, "quantize: negative shape");
  if (dtype != FDLLM_BF16 && dtype != FDLLM_F32) return fail(FDLLM_EINVAL, "quantize: bad dtype %d", dtype);
  if (rows == 0 || cols == 0) return FDLLM_OK;
  if (!src || !q || !scale) return fail(FDLLM_EINVAL, "quantize: null pointer");
  return cuda_status(launch_quantize_fp8(src, dtype == FDLLM_BF16, rows, cols, q, scale, (cudaStream_t)stream),
                     "quantize launch");
}

static fdllm_status resolve_select_fp8w(const fdllm_select_desc *desc, SelectProblem &p) {
  fdllm_status st = resolve_select(desc, p);
  if (st != FDLLM_OK) return st;
  p.fp8w = 1;
  if (!p.in_bf16 || !lmhead_tc_supported(p))
    return fail(FDLLM_EUNSUPPORTED,
                "select fp8w: needs bf16 hidden rows, hidden a multiple of 128 and batch * block_size <= 512");
  return FDLLM_OK;
}

size_t fdllm_select_fp8w_workspace_size(const fdllm_select_desc *desc) {
  SelectProblem p;
  if (resolve_select_fp8w(desc, p) != FDLLM_OK) return 0;
  return select_layout(p).total;
}

fdllm_status fdllm_confidence_select_fp8w(const fdllm_select_desc *desc, const void *hidden, const uint8_t *w_q,
                                          const float *w_scale, int32_t *tokens, uint8_t *unmasked, float *conf,
                                          float *kappa, int32_t *argmax, int32_t *n_masked_left, void *workspace,
                                          size_t ws_bytes, fdllm_stream_t stream) {
  SelectProblem p;
  fdllm_status st = resolve_select_fp8w(desc, p);
  if (st != FDLLM_OK) return st;
  const void *req[] = {hidden, w_q, w_scale, tokens, unmasked, conf, argmax, n_masked_left, workspace};
  const char *names[] = {"hidden", "w_q", "w_scale", "tokens", "unmasked", "conf", "argmax", "n_masked_left",
                         "workspace"};
  for (int i = 0; i < 9; ++i)
    if (!req[i]) return fail(FDLLM_EINVAL, "select fp8w: %s is null", names[i]);
  if (!aligned16(hidden) || !aligned16(w_q) || !aligned16(workspace))
    return fail(FDLLM_EINVAL, "select fp8w: hidden, w_q and workspace must be 16-byte aligned");
  const SelectLayout L = select_layout(p);
  if (ws_bytes < L.total)
    return fail(FDLLM_EINVAL, "select fp8w: workspace of %zu bytes is smaller than the %zu required", ws_bytes,
                L.total);
  st = check_cluster_operands(p, L.tc, workspace, w_q);   // the kernel reads the E4M3 rows from the workspace
  if (st != FDLLM_OK) return st;
  p.hidden = hidden; p.w = w_q; p.w_scale = w_scale; p.tokens = tokens; p.unmasked = unmasked; p.conf = conf;
  p.kappa = kappa; p.argmax = argmax; p.n_left = n_masked_left; p.ws = workspace; p.ws_bytes = ws_bytes;
  p.err = error_word_ptr();
  return cuda_status(run_select(p, L, workspace, (cudaStream_t)stream), "fp8 quantize / lm-head / select launch");
}

fdllm_status fdllm_block_attn_fp8kv(const fdllm_attn_desc *desc, const int32_t *block_idx, const void *q,
                                   const uint8_t *k_cache, const float *k_scale, const uint8_t *v_cache,
                                   const float *v_scale, const void *k_fresh, const void *v_fresh, void *out,
                                   float *lse, void *workspace, size_t ws_bytes, fdllm_stream_t stream) {
  if (!k_scale || !v_scale) return fail(FDLLM_EINVAL, "attn fp8kv: k_scale and v_scale are required");
  return block_attn(desc, block_idx, q, k_cache, v_cache, k_fresh, v_fresh, out, lse, workspace, ws_bytes, stream,
                    k_scale, v_scale);
}

fdllm_status fdllm_kv_splice_fp8(int32_t mode, int32_t batch, int32_t seq_len, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t start, int32_t len, int32_t src_dtype,
                                 uint8_t *k_cache, float *k_scale, uint8_t *v_cache, float *v_scale,
                                 const void *k_src, const void *v_src, fdllm_stream_t stream) {
  if (mode != FDLLM_SPLICE_WINDOW && mode != FDLLM_SPLICE_REFRESH)
    return fail(FDLLM_EINVAL, "splice fp8: unknown mode %d", mode);
  if (batch < 1 || seq_len < 1 || n_kv_heads < 1 || head_dim < 1)
    return fail(FDLLM_EINVAL, "splice fp8: batch, seq_len, n_kv_heads and head_dim must be >= 1");
  if (src_dtype != FDLLM_BF16 && src_dtype != FDLLM_F32)
    return fail(FDLLM_EINVAL, "splice fp8: bad source dtype %d", src_dtype);
  if (start < 0 || len < 0 || (int64_t)start + len > seq_len)
    return fail(FDLLM_EINVAL, "splice fp8: window [%d, %d) outside [0, %d)", start, start + len, seq_len);
  if (mode == FDLLM_SPLICE_REFRESH && (start != 0 || len != seq_len))
    return fail(FDLLM_EINVAL, "splice fp8: REFRESH rewrites the whole cache (start 0, len seq_len)");
  const void *ptrs[] = {k_cache, k_scale, v_cache, v_scale, k_src, v_src};
  for (int i = 0; i < 6; ++i)
    if (!ptrs[i]) return fail(FDLLM_EINVAL, "splice fp8: null pointer");
  if (len == 0) return FDLLM_OK;
  // one row per (sequence, position, KV head): source rows b * len * Hkv + i, cache rows
  // (b * seq_len + start) * Hkv + i
  const int64_t rpb = (int64_t)len * n_kv_heads, dst = (int64_t)seq_len * n_kv_heads;
  const int64_t off = (int64_t)start * n_kv_heads;
  const bool bf16 = src_dtype == FDLLM_BF16;
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = launch_quantize_fp8_batched(k_src, bf16, batch, rpb, head_dim, rpb, k_cache + off * head_dim,
                                              k_scale + off, dst, cs);
  if (e == cudaSuccess)
    e = launch_quantize_fp8_batched(v_src, bf16, batch, rpb, head_dim, rpb, v_cache + off * head_dim,
                                    v_scale + off, dst, cs);
  return cuda_status(e, "splice fp8 launch");
}

fdllm_status fdllm_kv_splice_fp8_ragged(int32_t batch, int32_t seq_len, int32_t n_kv_heads, int32_t head_dim,
                                        const int32_t *start, int32_t len, int32_t src_dtype, uint8_t *k_cache,
                                        float *k_scale, uint8_t *v_cache, float *v_scale, const void *k_src,
                                        const void *v_src, fdllm_stream_t stream) {
  if (!start) return fail(FDLLM_EINVAL, "splice fp8: start is null");
  if (batch < 1 || seq_len < 1 || n_kv_heads < 1 || head_dim < 1)
    return fail(FDLLM_EINVAL, "splice fp8: batch, seq_len, n_kv_heads and head_dim must be >= 1");
  if (src_dtype != FDLLM_BF16 && src_dtype != FDLLM_F32)
    return fail(FDLLM_EINVAL, "splice fp8: bad source dtype %d", src_dtype);
  if (len < 0 || len > seq_len) return fail(FDLLM_EINVAL, "splice fp8: len %d outside [0, %d]", len, seq_len);
  const void *ptrs[] = {k_cache, k_scale, v_cache, v_scale, k_src, v_src};
  for (int i = 0; i < 6; ++i)
    if (!ptrs[i]) return fail(FDLLM_EINVAL, "splice fp8: null pointer");
  if (len == 0) return FDLLM_OK;
  // source rows b * len * Hkv + i; cache rows (b * seq_len + start[b]) * Hkv + i
  const int64_t rpb = (int64_t)len * n_kv_heads, dst = (int64_t)seq_len * n_kv_heads;
  const bool bf16 = src_dtype == FDLLM_BF16;
  cudaStream_t cs = (cudaStream_t)stream;
  int32_t *err = error_word_ptr();
  cudaError_t e = launch_quantize_fp8_batched(k_src, bf16, batch, rpb, head_dim, rpb, k_cache, k_scale, dst, cs,
                                              start, n_kv_heads, seq_len - len, err);
  if (e == cudaSuccess)
    e = launch_quantize_fp8_batched(v_src, bf16, batch, rpb, head_dim, rpb, v_cache, v_scale, dst, cs, start,
                                    n_kv_heads, seq_len - len, err);
  return cuda_status(e, "splice fp8 launch");
}

fdllm_status fdllm_kv_splice(int32_t mode, int32_t batch, int32_t seq_len, int32_t n_kv_heads,
                             int32_t head_dim, int32_t start, int32_t len, int32_t dtype,
                             void *k_cache, void *v_cache, const void *k_src, const void *v_src,
                             fdllm_stream_t stream) {
  if (mode != FDLLM_SPLICE_WINDOW && mode != FDLLM_SPLICE_REFRESH)
    return fail(FDLLM_EINVAL, "splice: unknown mode %d", mode);
  if (batch < 1 || seq_len < 1 || n_kv_heads < 1 || head_dim < 1)
    return fail(FDLLM_EINVAL, "splice: batch, seq_len, n_kv_heads and head_dim must be >= 1");
  if (dtype != FDLLM_BF16 && dtype != FDLLM_F32) return fail(FDLLM_EINVAL, "splice: bad dtype %d", dtype);
  if (start < 0 || len < 0 || (int64_t)start + len > seq_len)
    return fail(FDLLM_EINVAL, "splice: window [%d, %d) outside [0, %d)", start, start + len, seq_len);
  if (mode == FDLLM_SPLICE_REFRESH && (start != 0 || len != seq_len))
    return fail(FDLLM_EINVAL, "splice: REFRESH rewrites the whole cache (start 0, len seq_len)");
  const int64_t row_bytes = (int64_t)n_kv_heads * head_dim * (dtype == FDLLM_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0) return fail(FDLLM_EINVAL, "splice: Hkv * d * element size must be a multiple of 16 bytes");
  const void *ptrs[] = {k_cache, v_cache, k_src, v_src};
  for (int i = 0; i < 4; ++i) {
    if (!ptrs[i]) return fail(FDLLM_EINVAL, "splice: null pointer");
    if (!aligned16(ptrs[i])) return fail(FDLLM_EINVAL, "splice: pointers must be 16-byte aligned");
  }
  return cuda_status(launch_splice(batch, seq_len, row_bytes, start, len, k_cache, v_cache, k_src,
                                   v_src, (cudaStream_t)stream),
                     "splice launch");
}

fdllm_status fdllm_kv_splice_ragged(int32_t batch, int32_t seq_len, int32_t n_kv_heads, int32_t head_dim,
                                    const int32_t *start, int32_t len, int32_t dtype, void *k_cache,
                                    void *v_cache, const void *k_src, const void *v_src, fdllm_stream_t stream) {
  if (!start) return fail(FDLLM_EINVAL, "splice: start is null");
  if (batch < 1 || seq_len < 1 || n_kv_heads < 1 || head_dim < 1)
    return fail(FDLLM_EINVAL, "splice: batch, seq_len, n_kv_heads and head_dim must be >= 1");
  if (dtype != FDLLM_BF16 && dtype != FDLLM_F32) return fail(FDLLM_EINVAL, "splice: bad dtype %d", dtype);
  if (len < 0 || len > seq_len) return fail(FDLLM_EINVAL, "splice: len %d outside [0, %d]", len, seq_len);
  const int64_t row_bytes = (int64_t)n_kv_heads * head_dim * (dtype == FDLLM_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0) return fail(FDLLM_EINVAL, "splice: Hkv * d * element size must be a multiple of 16 bytes");
  const void *ptrs[] = {k_cache, v_cache, k_src, v_src};
  for (int i = 0; i < 4; ++i) {
    if (!ptrs[i]) return fail(FDLLM_EINVAL, "splice: null pointer");
    if (!aligned16(ptrs[i])) return fail(FDLLM_EINVAL, "splice: pointers must be 16-byte aligned");
  }
  return cuda_status(launch_splice(batch, seq_len, row_bytes, 0, len, k_cache, v_cache, k_src, v_src,
                                   (cudaStream_t)stream, start, error_word_ptr()),
                     "splice launch");
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Allocation-free confidence select: the partials live in a file-scope device
// array instead of a caller workspace (see fdllm_confidence_select_noalloc in
// include/fdllm.h for the callers this serves and the limits).
// ----------------------------------------------------------------------------
namespace fdllm {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FDLLM_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a stand-in for the symbol, so the address is looked up
// once per device and context (with that device current) and cached; a new
// context on the device (after a device reset) gets a fresh lookup.
fdllm_status noalloc_scratch(void **out) {
  static SymbolCache cache;
  return cuda_status(cache.get((const void *)g_noalloc_scratch, out), "noalloc select: cudaGetSymbolAddress");
}

}  // namespace
}  // namespace fdllm

extern "C" fdllm_status fdllm_confidence_select_noalloc(const fdllm_select_desc *desc, const void *hidden,
                                                        const void *lm_head_w, int32_t *tokens,
                                                        uint8_t *unmasked, float *conf, float *kappa,
                                                        int32_t *argmax, int32_t *n_masked_left,
                                                        fdllm_stream_t stream) {
  SelectProblem p;
  fdllm_status st = resolve_select(desc, p);
  if (st != FDLLM_OK) return st;
  const void *req[] = {hidden, lm_head_w, tokens, unmasked, conf, argmax, n_masked_left};
  const char *names[] = {"hidden", "lm_head_w", "tokens", "unmasked", "conf", "argmax", "n_masked_left"};
  for (int i = 0; i < 7; ++i)
    if (!req[i]) return fail(FDLLM_EINVAL, "noalloc select: %s is null", names[i]);
  if (!aligned16(hidden) || !aligned16(lm_head_w))
    return fail(FDLLM_EINVAL, "noalloc select: hidden and lm_head_w must be 16-byte aligned");
  const SelectLayout L = select_layout(p);
  if (L.total > FDLLM_NOALLOC_SCRATCH_BYTES)
    return fail(FDLLM_EINVAL,
                "noalloc select: the vocabulary partials need %zu bytes, more than the %u-byte static scratch "
                "(batch * block_size = %d rows x %d splits); use fdllm_confidence_select with a workspace",
                L.total, (unsigned)FDLLM_NOALLOC_SCRATCH_BYTES, p.batch * p.B, L.splits);
  st = check_cluster_operands(p, L.tc, hidden, lm_head_w);
  if (st != FDLLM_OK) return st;
  void *scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != FDLLM_OK) return st;
  p.hidden = hidden; p.w = lm_head_w; p.tokens = tokens; p.unmasked = unmasked; p.conf = conf;
  p.kappa = kappa; p.argmax = argmax; p.n_left = n_masked_left;
  p.ws = scratch; p.ws_bytes = FDLLM_NOALLOC_SCRATCH_BYTES;
  p.err = error_word_ptr();
  return cuda_status(run_select(p, L, scratch, (cudaStream_t)stream), "noalloc select: lm-head / select launch");
}
