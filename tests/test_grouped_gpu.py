"""pa_decode_grouped (shared-prefix "cascade" decode) against the fp64 oracle
and against pa_decode on the same inputs.  The oracle knows nothing of
groups: sharing must not change the result."""
import numpy as np
import pytest
import torch

import gpu_util as U
from paged_kv_cache_blocks_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def run_grouped(pa, b, off=None, pre=None, ws=None):
    q, kc, vc, tab, lens = U.device_inputs(b)
    o, p = b.group_arrays()
    off = o if off is None else np.asarray(off, np.int32)
    pre = p if pre is None else np.asarray(pre, np.int32)
    if ws is None:
        ws = torch.empty(pa.pa_decode_grouped_workspace_bytes(len(b.seq_lens), q.shape[1], q.shape[2],
                                                              tab.shape[1] * 16),
                         dtype=torch.uint8, device="cuda")
    out = pa.pa_decode_grouped(q, kc, vc, tab, lens, b.workload.scale, torch.from_numpy(off).cuda(),
                               torch.from_numpy(pre).cuda(), workspace=ws)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), pa.pa_decode_check(ws)


def test_fullstep_groups(pa):
    b = U.batch("fullstep", num_layers=1)
    got, bits = run_grouped(pa, b)
    assert bits == 0
    U.assert_close(got, U.oracle_out_cached("fullstep", num_layers=1), "fullstep grouped")
    q, kc, vc, tab, lens = U.device_inputs(b)
    plain = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale).double().cpu().numpy()
    assert np.max(np.abs(got - plain)) <= 1e-2


def _mixed_batch(name, seed, groups, lens):
    return W.make_batch(name, seed=seed, lens_override=lens, groups=groups)


def test_edge_groups_g4(pa):
    rng = np.random.default_rng(9)
    groups = [(3, 32), (1, 16), (1, 0), (40, 1040), (5, 2048)]
    lens = [40, 33, 32, 100, 5] + list(rng.integers(1041, 1101, 40)) + [2048, 2049, 2600, 4000, 6000]
    b = _mixed_batch("llama8b", 21, groups, lens)
    got, bits = run_grouped(pa, b)
    assert bits == 0
    U.assert_close(got, U.oracle_out(b), "edge groups G=4")


def test_groups_g8_two_row_tiles(pa):
    rng = np.random.default_rng(10)
    groups = [(20, 512), (2, 0), (3, 1024)]
    lens = list(rng.integers(600, 801, 20)) + [7, 900] + [1024, 1500, 3000]
    b = _mixed_batch("llama70b", 22, groups, lens)
    got, bits = run_grouped(pa, b)
    assert bits == 0
    U.assert_close(got, U.oracle_out(b), "groups G=8")


def test_fp16_d64_groups(pa):
    b = _mixed_batch("tiny", 23, [(2, 16), (2, 0)], [17, 33, 1, 100])
    got, bits = run_grouped(pa, b)
    assert bits == 0
    U.assert_close(got, U.oracle_out(b), "groups fp16 d64")


def test_invalid_groups_are_flagged_and_still_correct(pa):
    rng = np.random.default_rng(11)
    lens = list(rng.integers(200, 400, 6))
    b = _mixed_batch("llama8b", 24, [(3, 128), (3, 64)], lens)
    ref = U.oracle_out(b)
    # a prefix that is not whole blocks
    got, bits = run_grouped(pa, b, pre=[120, 64])
    assert bits & pa.PA_DEVERR_GROUP
    U.assert_close(got, ref, "prefix not whole blocks")
    # offsets that do not cover the batch
    got, bits = run_grouped(pa, b, off=[0, 3, 5])
    assert bits & pa.PA_DEVERR_GROUP
    U.assert_close(got, ref, "bad offsets")
    # and a clean call afterwards on the same workspace
    got, bits = run_grouped(pa, b)
    assert bits == 0
    U.assert_close(got, ref, "clean")
