"""Failure detection on the GPU without a fault: the bounded mbarrier wait the
kernels use gives up after its limit, reports PA_DEVERR_TIMEOUT, and the
context stays usable (a decode right after is correct)."""
import time

import numpy as np
import pytest
import torch

import gpu_util as U

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_survives():
    pa = U.require_gpu()
    t0 = time.perf_counter()
    ok, err, abort, waited_us = pa.pa_selftest_bounded_wait(50_000_000)   # 50 ms
    elapsed = time.perf_counter() - t0
    assert ok == 0 and abort == 1
    assert err & pa.PA_DEVERR_TIMEOUT
    assert 50_000 <= waited_us < 1_000_000 and elapsed < 10
    # the context is intact: a decode afterwards matches the oracle
    b = U.batch("tiny")
    q, kc, vc, tab, lens = U.device_inputs(b)
    out = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale)
    torch.cuda.synchronize()
    U.assert_close(out.double().cpu().numpy(), U.oracle_out(b), "after the timeout")
