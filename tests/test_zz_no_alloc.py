"""pa_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (its scratch is a static 64 MiB array in libpa).

It must give the same output as pa_decode with a caller-provided workspace,
and stay within the decode tolerance of the fp64 oracle, on two calls in a
row (the static scratch keeps the previous call's contents, which the next
call must not depend on).  This file is collected last so that a failure
here never hides the other tests."""
import numpy as np
import pytest
import torch

import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def test_noalloc_matches_pa_decode_twice(pa):
    for name, seed in (("llama8b", 3), ("tiny", 0)):
        b = U.batch(name, seed=seed)
        q, kc, vc, tab, lens = U.device_inputs(b)
        ref = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale)
        torch.cuda.synchronize()
        ref = ref.double().cpu().numpy()
        exact = U.oracle_out(b)
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            pa.pa_decode_noalloc(q, kc, vc, tab, lens, b.workload.scale, out=out)
            torch.cuda.synchronize()
            got = out.double().cpu().numpy()
            assert np.isfinite(got).all()
            err = np.abs(got - ref)
            assert err.max() <= U.MAX_ABS and err.mean() <= U.MEAN_ABS, (name, err.max())
            U.assert_close(got, exact, f"noalloc {name} vs oracle")


def test_noalloc_rejects_batches_beyond_its_scratch(pa):
    b = U.batch("tiny")
    q, kc, vc, tab, lens = U.device_inputs(b)
    # 256 sequences of up to 1M tokens need far more than 64 MiB of partials
    qb = torch.zeros((256, 64, 128), dtype=torch.bfloat16, device="cuda")
    tb = torch.zeros((256, 65536), dtype=torch.int32, device="cuda")
    lb = torch.ones(256, dtype=torch.int32, device="cuda")
    kb = torch.zeros((4, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_noalloc(qb, kb, kb, tb, lb, 0.1)
    assert e.value.code == pa.PA_ERR_INVALID and "64 MiB" in str(e.value)
