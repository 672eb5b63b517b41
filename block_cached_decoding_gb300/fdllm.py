"""ctypes binding of libfdllm.so (include/fdllm.h, include/fdllm_synth.h).

Argument marshalling only: each function takes torch tensors (or raw device
addresses as ints) and forwards their addresses, sizes and the CUDA stream to
the C ABI of the same name; every step of the computation runs in the CUDA
library.  Loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfdllm.so")

OK, EINVAL, ECUDA, ETIMEOUT, EUNSUPPORTED = range(5)
BF16, F32 = 0, 1
SELECT_THRESHOLD, SELECT_FACTOR, SELECT_TOPK = 0, 1, 2
SPLICE_WINDOW, SPLICE_REFRESH = 0, 1
SYNTH_W, SYNTH_KCACHE, SYNTH_VCACHE, SYNTH_Q, SYNTH_KFRESH, SYNTH_VFRESH, SYNTH_HID, SYNTH_PLANT, SYNTH_PROMPT = range(1, 10)

EXPORTS = (
    "fdllm_attn_query_count", "fdllm_attn_workspace_size", "fdllm_block_attn",
    "fdllm_select_workspace_size", "fdllm_confidence_select", "fdllm_kv_splice",
    "fdllm_status_string", "fdllm_last_error", "fdllm_last_device_error", "fdllm_version",
    "fdllm_synth_normals", "fdllm_synth_kv_cache", "fdllm_synth_rows", "fdllm_synth_hidden",
    "fdllm_synth_prompt", "fdllm_launch_counter", "fdllm_confidence_select_noalloc",
    "fdllm_selftest_bounded_wait", "fdllm_block_attn_ragged", "fdllm_confidence_select_ragged",
    "fdllm_kv_splice_ragged", "fdllm_quantize_fp8_rows", "fdllm_select_fp8w_workspace_size",
    "fdllm_confidence_select_fp8w", "fdllm_block_attn_fp8kv", "fdllm_kv_splice_fp8", "fdllm_block_loop_create",
    "fdllm_block_loop_launch", "fdllm_block_loop_destroy", "fdllm_synth_rows_at", "fdllm_synth_hidden_at",
    "fdllm_kv_splice_fp8_ragged", "fdllm_block_attn_update", "fdllm_block_loop_create_refresh",
    "fdllm_synth_kv_cache_at", "fdllm_block_loop_create_ragged", "fdllm_synth_rows_seq", "fdllm_synth_hidden_seq",
    "fdllm_synth_kv_cache_seq",
)

# void step(void *user, fdllm_stream_t stream)
STEP_FN = C.CFUNCTYPE(None, C.c_void_p, C.c_void_p)

NOALLOC_SCRATCH_BYTES = 2 << 20


class FdllmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class AttnDesc(C.Structure):
    _fields_ = [("batch", C.c_int32), ("prompt_len", C.c_int32), ("gen_length", C.c_int32),
                ("block_size", C.c_int32), ("block_idx", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("use_cache", C.c_int32),
                ("dual_cache", C.c_int32), ("sm_scale", C.c_float), ("dtype", C.c_int32),
                ("out_f32", C.c_int32)]


class SelectDesc(C.Structure):
    _fields_ = [("batch", C.c_int32), ("seq_len", C.c_int32), ("block_start", C.c_int32),
                ("block_size", C.c_int32), ("hidden", C.c_int32), ("vocab", C.c_int32),
                ("mask_id", C.c_int32), ("strategy", C.c_int32), ("threshold", C.c_float),
                ("factor", C.c_float), ("topk", C.c_int32), ("dtype", C.c_int32)]


_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it is missing (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        L.fdllm_attn_query_count.argtypes = [C.POINTER(AttnDesc)]
        L.fdllm_attn_query_count.restype = i64
        L.fdllm_attn_workspace_size.argtypes = [C.POINTER(AttnDesc)]
        L.fdllm_attn_workspace_size.restype = sz
        L.fdllm_block_attn.argtypes = [C.POINTER(AttnDesc), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fdllm_block_attn.restype = i32
        L.fdllm_select_workspace_size.argtypes = [C.POINTER(SelectDesc)]
        L.fdllm_select_workspace_size.restype = sz
        L.fdllm_confidence_select.argtypes = [C.POINTER(SelectDesc)] + [vp] * 9 + [sz, vp]
        L.fdllm_confidence_select.restype = i32
        L.fdllm_confidence_select_noalloc.argtypes = [C.POINTER(SelectDesc)] + [vp] * 9
        L.fdllm_confidence_select_noalloc.restype = i32
        L.fdllm_kv_splice.argtypes = [i32] * 8 + [vp] * 5
        L.fdllm_kv_splice.restype = i32
        L.fdllm_block_attn_ragged.argtypes = [C.POINTER(AttnDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fdllm_block_attn_ragged.restype = i32
        L.fdllm_block_attn_update.argtypes = [C.POINTER(AttnDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fdllm_block_attn_update.restype = i32
        L.fdllm_confidence_select_ragged.argtypes = [C.POINTER(SelectDesc)] + [vp] * 10 + [sz, vp]
        L.fdllm_confidence_select_ragged.restype = i32
        L.fdllm_kv_splice_ragged.argtypes = [i32] * 4 + [vp, i32, i32] + [vp] * 5
        L.fdllm_kv_splice_ragged.restype = i32
        L.fdllm_quantize_fp8_rows.argtypes = [i64, i32, i32, vp, vp, vp, vp]
        L.fdllm_quantize_fp8_rows.restype = i32
        L.fdllm_select_fp8w_workspace_size.argtypes = [C.POINTER(SelectDesc)]
        L.fdllm_select_fp8w_workspace_size.restype = sz
        L.fdllm_confidence_select_fp8w.argtypes = [C.POINTER(SelectDesc)] + [vp] * 10 + [sz, vp]
        L.fdllm_confidence_select_fp8w.restype = i32
        L.fdllm_block_attn_fp8kv.argtypes = [C.POINTER(AttnDesc)] + [vp] * 11 + [sz, vp]
        L.fdllm_block_attn_fp8kv.restype = i32
        L.fdllm_kv_splice_fp8.argtypes = [i32] * 8 + [vp] * 7
        L.fdllm_kv_splice_fp8.restype = i32
        L.fdllm_kv_splice_fp8_ragged.argtypes = [i32] * 4 + [vp, i32, i32] + [vp] * 7
        L.fdllm_kv_splice_fp8_ragged.restype = i32
        L.fdllm_status_string.argtypes = [i32]
        L.fdllm_status_string.restype = C.c_char_p
        L.fdllm_last_error.argtypes = []
        L.fdllm_last_error.restype = C.c_char_p
        L.fdllm_last_device_error.argtypes = [vp, C.POINTER(i32)]
        L.fdllm_last_device_error.restype = i32
        L.fdllm_version.argtypes = []
        L.fdllm_version.restype = i32
        L.fdllm_selftest_bounded_wait.argtypes = [i32, vp]
        L.fdllm_selftest_bounded_wait.restype = i32
        L.fdllm_launch_counter.argtypes = []
        L.fdllm_launch_counter.restype = C.c_uint64
        u64 = C.c_uint64
        L.fdllm_synth_normals.argtypes = [u64, i32, C.POINTER(i64), i32, i64, i64, C.c_float, i32, vp, vp]
        L.fdllm_synth_kv_cache.argtypes = [u64, i32, i32, i32, i32, i32, i64, C.c_float, i32, vp, vp]
        L.fdllm_synth_rows.argtypes = [u64, i32, i32, i64, i32, i32, i32, C.c_float, i32, vp, vp]
        L.fdllm_synth_hidden.argtypes = [u64, i32, i64, i32, i32, i32, i32, C.c_double, vp, i32, vp, vp]
        L.fdllm_synth_prompt.argtypes = [u64, i32, i32, i32, vp, vp]
        L.fdllm_synth_rows_at.argtypes = [u64, i32, i32, i64, vp, i32, i32, i32, C.c_float, i32, vp, vp]
        L.fdllm_synth_hidden_at.argtypes = [u64, i32, i64, vp, i32, i32, i32, i32, C.c_double, vp, i32, vp, vp]
        L.fdllm_block_loop_create.argtypes = [C.POINTER(vp), STEP_FN, vp, vp, i32, i32, vp, vp]
        L.fdllm_block_loop_create.restype = i32
        L.fdllm_block_loop_create_refresh.argtypes = [C.POINTER(vp), STEP_FN, STEP_FN, vp, vp, i32, i32, i32, vp, vp]
        L.fdllm_block_loop_create_refresh.restype = i32
        L.fdllm_synth_kv_cache_at.argtypes = [u64, i32, i32, i32, i32, i32, i64, vp, i64, C.c_float, i32, vp, vp]
        L.fdllm_block_loop_create_ragged.argtypes = [C.POINTER(vp), STEP_FN, STEP_FN, vp, vp, i32, i32, i32, i32,
                                                     vp, vp, vp, vp, vp, vp, vp]
        L.fdllm_block_loop_create_ragged.restype = i32
        L.fdllm_synth_rows_seq.argtypes = [u64, i32, i32, vp, vp, i32, i32, C.c_float, i32, vp, vp]
        L.fdllm_synth_hidden_seq.argtypes = [u64, i32, vp, vp, i32, i32, i32, C.c_double, vp, i32, vp, vp]
        L.fdllm_synth_kv_cache_seq.argtypes = [u64, i32, i32, i32, i32, i32, vp, vp, C.c_float, i32, vp, vp]
        L.fdllm_block_loop_launch.argtypes = [vp, vp]
        L.fdllm_block_loop_launch.restype = i32
        L.fdllm_block_loop_destroy.argtypes = [vp]
        L.fdllm_block_loop_destroy.restype = None
        for f in ("fdllm_synth_normals", "fdllm_synth_kv_cache", "fdllm_synth_rows", "fdllm_synth_hidden",
                  "fdllm_synth_prompt", "fdllm_synth_rows_at", "fdllm_synth_hidden_at", "fdllm_synth_kv_cache_at",
                  "fdllm_synth_rows_seq", "fdllm_synth_hidden_seq", "fdllm_synth_kv_cache_seq"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int):
    if st != OK:
        msg = lib().fdllm_last_error().decode(errors="replace")
        raise FdllmError(st, msg or lib().fdllm_status_string(st).decode())


def dtype_code(t) -> int:
    import torch
    return {torch.bfloat16: BF16, torch.float32: F32}[t.dtype]


# ---------------------------------------------------------------------------
# hot path
# ---------------------------------------------------------------------------

def attn_desc(*, batch, prompt_len, gen_length, block_size, block_idx, n_q_heads, n_kv_heads, head_dim,
              use_cache=1, dual_cache=1, sm_scale=0.0, dtype=BF16, out_f32=1) -> AttnDesc:
    return AttnDesc(batch, prompt_len, gen_length, block_size, block_idx, n_q_heads, n_kv_heads, head_dim,
                    use_cache, dual_cache, sm_scale, dtype, out_f32)


def select_desc(*, batch, seq_len, block_start, block_size, hidden, vocab, mask_id, threshold=0.9,
                strategy=SELECT_THRESHOLD, factor=1.0, topk=1, dtype=BF16) -> SelectDesc:
    return SelectDesc(batch, seq_len, block_start, block_size, hidden, vocab, mask_id, strategy, threshold,
                      factor, topk, dtype)


def fdllm_attn_query_count(desc: AttnDesc) -> int:
    return lib().fdllm_attn_query_count(C.byref(desc))


def fdllm_attn_workspace_size(desc: AttnDesc) -> int:
    return lib().fdllm_attn_workspace_size(C.byref(desc))


def fdllm_block_attn(desc, q, k_cache, v_cache, k_fresh, v_fresh, out, lse=None, workspace=None,
                     ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fdllm_block_attn(C.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_fresh),
                                  _ptr(v_fresh), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                  _stream(stream)))


def fdllm_select_workspace_size(desc: SelectDesc) -> int:
    return lib().fdllm_select_workspace_size(C.byref(desc))


def fdllm_select_fp8w_workspace_size(desc: SelectDesc) -> int:
    return lib().fdllm_select_fp8w_workspace_size(C.byref(desc))


def fdllm_quantize_fp8_rows(rows, cols, dtype, src, q, scale, stream=None):
    """Per-row E4M3 codes q [rows, cols] (uint8) and power-of-two scales [rows] (fp32) of src."""
    _check(lib().fdllm_quantize_fp8_rows(rows, cols, dtype, _ptr(src), _ptr(q), _ptr(scale), _stream(stream)))


def fdllm_confidence_select_fp8w(desc, hidden, w_q, w_scale, tokens, unmasked, conf, kappa, argmax, n_masked_left,
                                 workspace, ws_bytes=None, stream=None):
    """fdllm_confidence_select with the LM-head weight from the FP8 cache (w_q codes, w_scale per row)."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fdllm_confidence_select_fp8w(C.byref(desc), _ptr(hidden), _ptr(w_q), _ptr(w_scale), _ptr(tokens),
                                              _ptr(unmasked), _ptr(conf), _ptr(kappa), _ptr(argmax),
                                              _ptr(n_masked_left), _ptr(workspace), ws_bytes, _stream(stream)))


def fdllm_confidence_select(desc, hidden, lm_head_w, tokens, unmasked, conf, kappa, argmax, n_masked_left,
                            workspace, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fdllm_confidence_select(C.byref(desc), _ptr(hidden), _ptr(lm_head_w), _ptr(tokens),
                                         _ptr(unmasked), _ptr(conf), _ptr(kappa), _ptr(argmax),
                                         _ptr(n_masked_left), _ptr(workspace), ws_bytes, _stream(stream)))


def fdllm_confidence_select_noalloc(desc, hidden, lm_head_w, tokens, unmasked, conf, kappa, argmax, n_masked_left,
                                    stream=None):
    """fdllm_confidence_select with its scratch in the library's static device array (no workspace)."""
    _check(lib().fdllm_confidence_select_noalloc(C.byref(desc), _ptr(hidden), _ptr(lm_head_w), _ptr(tokens),
                                                 _ptr(unmasked), _ptr(conf), _ptr(kappa), _ptr(argmax),
                                                 _ptr(n_masked_left), _stream(stream)))


def fdllm_kv_splice(mode, batch, seq_len, n_kv_heads, head_dim, start, length, dtype, k_cache, v_cache,
                    k_src, v_src, stream=None):
    _check(lib().fdllm_kv_splice(mode, batch, seq_len, n_kv_heads, head_dim, start, length, dtype,
                                 _ptr(k_cache), _ptr(v_cache), _ptr(k_src), _ptr(v_src), _stream(stream)))


def fdllm_block_attn_ragged(desc, block_idx, q, k_cache, v_cache, k_fresh, v_fresh, out, lse=None,
                            workspace=None, ws_bytes=None, stream=None):
    """fdllm_block_attn (DualCache) with sequence b at block block_idx[b] (device int32 [batch])."""
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fdllm_block_attn_ragged(C.byref(desc), _ptr(block_idx), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(k_fresh), _ptr(v_fresh), _ptr(out), _ptr(lse), _ptr(workspace),
                                         ws_bytes, _stream(stream)))


def fdllm_block_attn_update(desc, block_idx, q, k_cache, v_cache, k_fresh, v_fresh, out, lse=None,
                            workspace=None, ws_bytes=None, stream=None):
    """fdllm_block_attn (block_idx None) or its per-sequence form, plus the cache-window update: cache rows
    [s_b, s_b + block_size) <- the block's fresh K/V."""
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fdllm_block_attn_update(C.byref(desc), _ptr(block_idx), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(k_fresh), _ptr(v_fresh), _ptr(out), _ptr(lse), _ptr(workspace),
                                         ws_bytes, _stream(stream)))


def fdllm_confidence_select_ragged(desc, block_start, hidden, lm_head_w, tokens, unmasked, conf, kappa, argmax,
                                   n_masked_left, workspace, ws_bytes=None, stream=None):
    """fdllm_confidence_select with sequence b's block at block_start[b] (device int32 [batch])."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fdllm_confidence_select_ragged(C.byref(desc), _ptr(block_start), _ptr(hidden), _ptr(lm_head_w),
                                                _ptr(tokens), _ptr(unmasked), _ptr(conf), _ptr(kappa),
                                                _ptr(argmax), _ptr(n_masked_left), _ptr(workspace), ws_bytes,
                                                _stream(stream)))


def fdllm_kv_splice_ragged(batch, seq_len, n_kv_heads, head_dim, start, length, dtype, k_cache, v_cache,
                           k_src, v_src, stream=None):
    """Window splice with sequence b's window at start[b] (device int32 [batch])."""
    _check(lib().fdllm_kv_splice_ragged(batch, seq_len, n_kv_heads, head_dim, _ptr(start), length, dtype,
                                        _ptr(k_cache), _ptr(v_cache), _ptr(k_src), _ptr(v_src), _stream(stream)))


def fdllm_block_attn_fp8kv(desc, block_idx, q, k_cache, k_scale, v_cache, v_scale, k_fresh, v_fresh, out, lse=None,
                           workspace=None, ws_bytes=None, stream=None):
    """fdllm_block_attn over an FP8 cache (E4M3 codes + per-row scales); block_idx None or device int32 [batch]."""
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fdllm_block_attn_fp8kv(C.byref(desc), _ptr(block_idx), _ptr(q), _ptr(k_cache), _ptr(k_scale),
                                        _ptr(v_cache), _ptr(v_scale), _ptr(k_fresh), _ptr(v_fresh), _ptr(out),
                                        _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))


def fdllm_kv_splice_fp8(mode, batch, seq_len, n_kv_heads, head_dim, start, length, src_dtype, k_cache, k_scale,
                        v_cache, v_scale, k_src, v_src, stream=None):
    """Quantise src rows into the FP8 cache window [start, start + length)."""
    _check(lib().fdllm_kv_splice_fp8(mode, batch, seq_len, n_kv_heads, head_dim, start, length, src_dtype,
                                     _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale), _ptr(k_src),
                                     _ptr(v_src), _stream(stream)))


def fdllm_kv_splice_fp8_ragged(batch, seq_len, n_kv_heads, head_dim, start, length, src_dtype, k_cache, k_scale,
                               v_cache, v_scale, k_src, v_src, stream=None):
    """Quantise src rows into each sequence's FP8 cache window at start[b] (device int32 [batch])."""
    _check(lib().fdllm_kv_splice_fp8_ragged(batch, seq_len, n_kv_heads, head_dim, _ptr(start), length, src_dtype,
                                            _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale), _ptr(k_src),
                                            _ptr(v_src), _stream(stream)))


def fdllm_last_device_error(stream=None) -> tuple[int, int]:
    detail = C.c_int32(0)
    st = lib().fdllm_last_device_error(_stream(stream), C.byref(detail))
    return st, detail.value


def fdllm_version() -> int:
    return lib().fdllm_version()


def fdllm_selftest_bounded_wait(limit_ms: int, stream=None):
    _check(lib().fdllm_selftest_bounded_wait(limit_ms, _stream(stream)))


def fdllm_launch_counter() -> int:
    return lib().fdllm_launch_counter()


# ---------------------------------------------------------------------------
# device twin of the seeded input generator (harness, not the method)
# ---------------------------------------------------------------------------

def fdllm_synth_normals(seed, kind, coords, n, offset, sigma, dtype, out, stream=None):
    arr = (C.c_int64 * max(1, len(coords)))(*coords)
    _check(lib().fdllm_synth_normals(seed, kind, arr, len(coords), n, offset, sigma, dtype, _ptr(out),
                                     _stream(stream)))


def fdllm_synth_kv_cache(seed, kind, batch, seq_len, n_kv_heads, head_dim, epoch, sigma, dtype, out, stream=None):
    _check(lib().fdllm_synth_kv_cache(seed, kind, batch, seq_len, n_kv_heads, head_dim, epoch, sigma, dtype,
                                      _ptr(out), _stream(stream)))


def fdllm_synth_kv_cache_at(seed, kind, batch, seq_len, n_kv_heads, head_dim, epoch, epoch_add, epoch_div, sigma,
                            dtype, out, stream=None):
    """fdllm_synth_kv_cache with the epoch epoch + *epoch_add // epoch_div (epoch_add: device int64)."""
    _check(lib().fdllm_synth_kv_cache_at(seed, kind, batch, seq_len, n_kv_heads, head_dim, epoch, _ptr(epoch_add),
                                         epoch_div, sigma, dtype, _ptr(out), _stream(stream)))


def fdllm_synth_rows(seed, kind, batch, step, pos0, npos, width, sigma, dtype, out, stream=None):
    _check(lib().fdllm_synth_rows(seed, kind, batch, step, pos0, npos, width, sigma, dtype, _ptr(out),
                                  _stream(stream)))


def fdllm_synth_hidden(seed, batch, step, pos0, npos, hidden, vocab, p_plant, w, dtype, out, stream=None):
    _check(lib().fdllm_synth_hidden(seed, batch, step, pos0, npos, hidden, vocab, p_plant, _ptr(w), dtype,
                                    _ptr(out), _stream(stream)))


def fdllm_synth_rows_at(seed, kind, batch, step, step_add, pos0, npos, width, sigma, dtype, out, stream=None):
    """fdllm_synth_rows at step + *step_add (step_add: a device int64 tensor, read when the kernel runs)."""
    _check(lib().fdllm_synth_rows_at(seed, kind, batch, step, _ptr(step_add), pos0, npos, width, sigma, dtype,
                                     _ptr(out), _stream(stream)))


def fdllm_synth_hidden_at(seed, batch, step, step_add, pos0, npos, hidden, vocab, p_plant, w, dtype, out,
                          stream=None):
    _check(lib().fdllm_synth_hidden_at(seed, batch, step, _ptr(step_add), pos0, npos, hidden, vocab, p_plant,
                                       _ptr(w), dtype, _ptr(out), _stream(stream)))


def fdllm_synth_rows_seq(seed, kind, batch, step, pos0, npos, width, sigma, dtype, out, stream=None):
    """fdllm_synth_rows with sequence b at step[b] and first position pos0[b] (device int32 [batch])."""
    _check(lib().fdllm_synth_rows_seq(seed, kind, batch, _ptr(step), _ptr(pos0), npos, width, sigma, dtype,
                                      _ptr(out), _stream(stream)))


def fdllm_synth_hidden_seq(seed, batch, step, pos0, npos, hidden, vocab, p_plant, w, dtype, out, stream=None):
    _check(lib().fdllm_synth_hidden_seq(seed, batch, _ptr(step), _ptr(pos0), npos, hidden, vocab, p_plant, _ptr(w),
                                        dtype, _ptr(out), _stream(stream)))


def fdllm_synth_kv_cache_seq(seed, kind, batch, seq_len, n_kv_heads, head_dim, epoch, only, sigma, dtype, out,
                             stream=None):
    """Cache rows of sequence b for epoch epoch[b] (device int32), only where only[b] (device uint8, or None)."""
    _check(lib().fdllm_synth_kv_cache_seq(seed, kind, batch, seq_len, n_kv_heads, head_dim, _ptr(epoch), _ptr(only),
                                          sigma, dtype, _ptr(out), _stream(stream)))


class BlockLoop:
    """fdllm_block_loop: `step(stream)` is captured once as the body of a device-side while-loop that runs
    until n_masked_left is all zero or max_steps steps have run; `counter` (device int64) counts them per
    launch, `total` (device int64 or None) across launches."""

    def __init__(self, step, n_masked_left, batch, max_steps, counter, total=None, refresh=None, refresh_every=0,
                 ragged=None):
        """With `refresh(stream)` and refresh_every = r, fdllm_block_loop_create_refresh: the captured refresh
        runs before step c of each launch whenever c > 0 and r divides c.  With `ragged` = dict(n_blocks,
        block_size, block_idx, block_start, seq_steps, refresh_flags, done) (device tensors),
        fdllm_block_loop_create_ragged: one loop over the whole per-sequence generation, `refresh(stream)`
        (optional) running whenever some sequence moved to its next block."""
        self._h = None
        errors = []

        def wrap(fn):
            def body(user, stream):
                try:
                    fn(stream)
                except BaseException as e:       # an exception cannot cross the C frame: keep it
                    errors.append(e)
            return body

        self._cb = STEP_FN(wrap(step))           # kept alive with the loop
        h = C.c_void_p()
        if ragged is not None:
            self._rcb = STEP_FN(wrap(refresh)) if refresh is not None else STEP_FN(0)
            st = lib().fdllm_block_loop_create_ragged(
                C.byref(h), self._cb, self._rcb, None, _ptr(n_masked_left), batch, ragged["n_blocks"],
                ragged["block_size"], max_steps, _ptr(ragged["block_idx"]), _ptr(ragged["block_start"]),
                _ptr(ragged["seq_steps"]), _ptr(ragged["refresh_flags"]), _ptr(ragged["done"]), _ptr(counter),
                _ptr(total))
        elif refresh is not None and refresh_every:
            self._rcb = STEP_FN(wrap(refresh))
            st = lib().fdllm_block_loop_create_refresh(C.byref(h), self._cb, self._rcb, None, _ptr(n_masked_left),
                                                       batch, max_steps, refresh_every, _ptr(counter), _ptr(total))
        else:
            st = lib().fdllm_block_loop_create(C.byref(h), self._cb, None, _ptr(n_masked_left), batch, max_steps,
                                               _ptr(counter), _ptr(total))
        if st == OK:
            self._h = h
        if errors:
            self.close()
            raise errors[0]
        _check(st)

    def launch(self, stream=None):
        _check(lib().fdllm_block_loop_launch(self._h, _stream(stream)))

    def close(self):
        if self._h:
            lib().fdllm_block_loop_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fdllm_synth_prompt(seed, batch, prompt_len, vocab, out, stream=None):
    _check(lib().fdllm_synth_prompt(seed, batch, prompt_len, vocab, _ptr(out), _stream(stream)))
