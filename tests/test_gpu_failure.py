"""Failure detection without a GPU fault: a bounded device wait that runs out
sets the device error word, the host reads FDLLM_ETIMEOUT, and the context
keeps working.  Nothing here traps, faults or hangs the GPU: the waited-on
barrier is simply never arrived at and the wait gives up after 20 ms."""
import time

import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def test_bounded_wait_reports_timeout_and_context_survives():
    assert F.fdllm_last_device_error() == (F.OK, 0)       # clean before
    t0 = time.time()
    F.fdllm_selftest_bounded_wait(20)
    st, site = F.fdllm_last_device_error()
    assert st == F.ETIMEOUT and site == 900
    assert time.time() - t0 < 5.0
    assert F.fdllm_last_device_error() == (F.OK, 0)       # reading clears the word
    # the context still runs kernels: a splice round-trip
    k = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    src = torch.ones(1, 2, 1, 64, dtype=torch.bfloat16, device="cuda")
    F.fdllm_kv_splice(F.SPLICE_WINDOW, 1, 8, 1, 64, 3, 2, F.BF16, k, v, src, src)
    torch.cuda.synchronize()
    assert torch.equal(k[0, 3:5], src[0]) and k[0, :3].abs().sum() == 0


def test_selftest_rejects_bad_limits():
    for bad in (0, 5000):
        with pytest.raises(F.FdllmError) as e:
            F.fdllm_selftest_bounded_wait(bad)
        assert e.value.status == F.EINVAL
