"""The C ABI library loads, exports every declared symbol and rejects bad
arguments on the host (no GPU needed: validation runs before any launch)."""
import ctypes as C
import glob
import os
import re

import pytest

from block_cached_decoding_gb300 import fdllm as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(fdllm_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(F.LIB_PATH):
        from block_cached_decoding_gb300 import build
        build.build()
    return F.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert {"fdllm_block_attn", "fdllm_confidence_select", "fdllm_kv_splice"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(F.EXPORTS) <= declared


def test_status_strings_and_version(lib):
    assert F.fdllm_version() == 106
    for s in range(5):
        assert lib.fdllm_status_string(s).decode().startswith("FDLLM_")


def _attn(**kw):
    base = dict(batch=1, prompt_len=64, gen_length=64, block_size=16, block_idx=0, n_q_heads=4, n_kv_heads=4,
                head_dim=64, use_cache=1, dual_cache=1, dtype=F.F32)
    base.update(kw)
    return F.attn_desc(**base)


def test_query_counts_follow_the_cache_mode(lib):
    # DualCache: the block; PrefixCache: block + suffix; no cache: every position
    assert F.fdllm_attn_query_count(_attn()) == 16
    assert F.fdllm_attn_query_count(_attn(dual_cache=0, block_idx=1)) == 128 - 80
    assert F.fdllm_attn_query_count(_attn(use_cache=0)) == 128


@pytest.mark.parametrize("bad", [dict(batch=0), dict(block_idx=4), dict(block_idx=-1), dict(gen_length=60),
                                 dict(n_q_heads=6), dict(head_dim=96), dict(use_cache=2), dict(dtype=7),
                                 dict(sm_scale=float("nan"))])
def test_attn_rejects_bad_descriptors(lib, bad):
    d = _attn(**bad)
    assert F.fdllm_attn_query_count(d) == -1
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_block_attn(d, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == F.EINVAL


def test_attn_rejects_null_and_misaligned_pointers(lib):
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_block_attn(_attn(), 16, 16, 0, 16, 16, 16, stream=0)
    assert e.value.status == F.EINVAL and "v_cache is null" in str(e.value)
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_block_attn(_attn(), 16, 18, 16, 16, 16, 16, stream=0)
    assert e.value.status == F.EINVAL and "aligned" in str(e.value)


def _sel(**kw):
    base = dict(batch=1, seq_len=128, block_start=64, block_size=16, hidden=256, vocab=1024, mask_id=1024,
                threshold=0.9, dtype=F.F32)
    base.update(kw)
    return F.select_desc(**base)


@pytest.mark.parametrize("bad", [dict(block_size=0), dict(block_size=300), dict(block_start=120),
                                 dict(hidden=100), dict(vocab=1), dict(mask_id=5), dict(strategy=9),
                                 dict(strategy=F.SELECT_FACTOR, factor=0.0), dict(strategy=F.SELECT_TOPK, topk=0),
                                 dict(threshold=float("nan")), dict(batch=16, block_size=256)])
def test_select_rejects_bad_descriptors(lib, bad):
    d = _sel(**bad)
    assert F.fdllm_select_workspace_size(d) == 0
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_confidence_select(d, 16, 16, 16, 16, 16, 16, 16, 16, 16, ws_bytes=1 << 30, stream=0)
    assert e.value.status == F.EINVAL


def test_select_rejects_short_workspace(lib):
    d = _sel()
    need = F.fdllm_select_workspace_size(d)
    assert need > 0
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_confidence_select(d, 16, 16, 16, 16, 16, 16, 16, 16, 16, ws_bytes=need - 1, stream=0)
    assert e.value.status == F.EINVAL and "workspace" in str(e.value)


@pytest.mark.parametrize("args", [
    (F.SPLICE_WINDOW, 1, 128, 4, 64, 120, 16),     # window past the end
    (F.SPLICE_REFRESH, 1, 128, 4, 64, 0, 64),      # refresh must cover the whole cache
    (F.SPLICE_WINDOW, 1, 128, 1, 4, 0, 16),        # row of 16 bytes fp32 ok, but 4 bf16 = 8 bytes
    (5, 1, 128, 4, 64, 0, 16),
])
def test_splice_rejects_bad_windows(lib, args):
    mode, b, n, hkv, d, start, ln = args
    dtype = F.BF16 if (hkv, d) == (1, 4) else F.F32
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_kv_splice(mode, b, n, hkv, d, start, ln, dtype, 16, 16, 16, 16, stream=0)
    assert e.value.status == F.EINVAL


def test_per_sequence_block_calls_validate_on_the_host(lib):
    """The per-sequence calls reject a missing index array and unsupported modes before any launch."""
    def st(fn, *args):
        return fn(*args)
    d = _attn(dtype=F.BF16, head_dim=128)
    v = C.c_void_p(16)                       # never dereferenced: validation fails first
    assert lib.fdllm_block_attn_ragged(C.byref(d), None, v, v, v, v, v, v, None, v, 1 << 20, None) == F.EINVAL
    fp32 = _attn()
    assert lib.fdllm_block_attn_ragged(C.byref(fp32), v, v, v, v, v, v, v, None, v, 1 << 20, None) == F.EUNSUPPORTED
    prefix = _attn(dtype=F.BF16, head_dim=128, dual_cache=0)
    assert lib.fdllm_block_attn_ragged(C.byref(prefix), v, v, v, v, v, v, v, None, v, 1 << 20, None) == F.EUNSUPPORTED
    sd = F.select_desc(batch=2, seq_len=64, block_start=0, block_size=16, hidden=128, vocab=100, mask_id=100)
    assert lib.fdllm_confidence_select_ragged(C.byref(sd), None, v, v, v, v, v, v, v, v, v, 1 << 20,
                                              None) == F.EINVAL
    assert lib.fdllm_kv_splice_ragged(2, 64, 4, 64, None, 16, F.BF16, v, v, v, v, None) == F.EINVAL
    assert lib.fdllm_kv_splice_ragged(2, 64, 4, 64, v, 65, F.BF16, v, v, v, v, None) == F.EINVAL


def test_fp8_calls_validate_on_the_host(lib):
    """The FP8 weight-cache calls reject unsupported descriptors and null pointers before any launch."""
    v = C.c_void_p(16)
    ok = F.select_desc(batch=1, seq_len=64, block_start=0, block_size=16, hidden=256, vocab=100, mask_id=100)
    for bad in (dict(hidden=192), dict(dtype=F.F32), dict(batch=40, block_size=16)):
        kw = dict(batch=1, seq_len=700, block_start=0, block_size=16, hidden=256, vocab=100, mask_id=100)
        kw.update(bad)
        d = F.select_desc(**kw)
        assert F.fdllm_select_fp8w_workspace_size(d) == 0
        assert lib.fdllm_confidence_select_fp8w(C.byref(d), v, v, v, v, v, v, v, v, v, v, 1 << 30,
                                                None) == F.EUNSUPPORTED
    assert lib.fdllm_confidence_select_fp8w(C.byref(ok), v, v, None, v, v, v, v, v, v, v, 1 << 30,
                                            None) == F.EINVAL
    assert lib.fdllm_quantize_fp8_rows(4, 64, 7, v, v, v, None) == F.EINVAL
    assert lib.fdllm_quantize_fp8_rows(-1, 64, F.BF16, v, v, v, None) == F.EINVAL
    assert lib.fdllm_quantize_fp8_rows(4, 64, F.BF16, None, v, v, None) == F.EINVAL
    assert lib.fdllm_quantize_fp8_rows(0, 64, F.BF16, None, None, None, None) == F.OK


def test_fp8kv_calls_validate_on_the_host(lib):
    """The FP8 KV cache calls reject a cache-free mode, fp32 descriptors and missing scales before any launch."""
    v = C.c_void_p(16)
    d = _attn(dtype=F.BF16, head_dim=128)
    assert lib.fdllm_block_attn_fp8kv(C.byref(d), None, v, v, None, v, v, v, v, v, None, v, 1 << 20,
                                      None) == F.EINVAL
    nocache = _attn(dtype=F.BF16, head_dim=128, use_cache=0)
    assert lib.fdllm_block_attn_fp8kv(C.byref(nocache), None, v, v, v, v, v, v, v, v, None, v, 1 << 20,
                                      None) == F.EUNSUPPORTED
    assert lib.fdllm_block_attn_fp8kv(C.byref(_attn()), None, v, v, v, v, v, v, v, v, None, v, 1 << 20,
                                      None) == F.EUNSUPPORTED
    assert lib.fdllm_kv_splice_fp8(F.SPLICE_WINDOW, 1, 64, 2, 64, 60, 8, F.BF16, v, v, v, v, v, v, None) == F.EINVAL
    assert lib.fdllm_kv_splice_fp8(F.SPLICE_REFRESH, 1, 64, 2, 64, 0, 32, F.BF16, v, v, v, v, v, v, None) == F.EINVAL
    assert lib.fdllm_kv_splice_fp8(F.SPLICE_WINDOW, 1, 64, 2, 64, 0, 8, 5, v, v, v, v, v, v, None) == F.EINVAL
    assert lib.fdllm_kv_splice_fp8(F.SPLICE_WINDOW, 1, 64, 2, 64, 0, 8, F.BF16, v, None, v, v, v, v,
                                   None) == F.EINVAL


def test_block_loop_validates_on_the_host(lib):
    """The device-driven loop rejects missing pointers and empty shapes before touching the device."""
    h = C.c_void_p()
    v = C.c_void_p(16)
    cb = F.STEP_FN(lambda user, stream: None)
    assert lib.fdllm_block_loop_create(C.byref(h), cb, None, None, 1, 4, v, None) == F.EINVAL
    assert lib.fdllm_block_loop_create(C.byref(h), cb, None, v, 0, 4, v, None) == F.EINVAL
    assert lib.fdllm_block_loop_create(C.byref(h), cb, None, v, 1, 0, v, None) == F.EINVAL
    assert lib.fdllm_block_loop_create(C.byref(h), cb, None, v, 1, 4, None, None) == F.EINVAL
    assert lib.fdllm_block_loop_launch(None, None) == F.EINVAL


def test_synth_generators_validate_on_the_host(lib):
    """The seeded input generators reject shapes their launch cannot cover (a row of more than
    65535 chunks of 512 elements, more than 65535 sequences) and missing pointers before any launch."""
    v = C.c_void_p(16)
    assert lib.fdllm_synth_rows(1, 2, 1, 0, 0, 4, 65535 * 512 + 1, 1.0, F.BF16, v, None) == F.EINVAL
    assert lib.fdllm_synth_rows(1, 2, 65536, 0, 0, 4, 64, 1.0, F.BF16, v, None) == F.EINVAL
    assert lib.fdllm_synth_rows(1, 2, 1, 0, 0, 4, 64, 1.0, 7, v, None) == F.EINVAL
    assert lib.fdllm_synth_rows(1, 2, 1, 0, 0, 4, 64, 1.0, F.BF16, None, None) == F.EINVAL
    assert lib.fdllm_synth_rows(1, 2, 1, 0, 0, 0, 64, 1.0, F.BF16, None, None) == F.OK   # nothing to draw
    assert lib.fdllm_synth_hidden(1, 1, 0, 0, 4, 65535 * 512 + 1, 100, 0.5, v, F.BF16, v, None) == F.EINVAL
    assert lib.fdllm_synth_hidden(1, 1, 0, 0, 4, 64, 100, -0.5, v, F.BF16, v, None) == F.EINVAL
    assert lib.fdllm_synth_hidden(1, 1, 0, 0, 4, 64, 100, 0.5, None, F.BF16, v, None) == F.EINVAL
