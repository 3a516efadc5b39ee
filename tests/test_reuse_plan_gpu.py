"""Plan reuse (PA_DECODE_REUSE_PLAN): the later layers of one decode step skip
the prep kernel and decode with the partition list the first layer's call
left in the workspace.  The outputs must be bit-identical to a full call and
within tolerance of the oracle, empty sequences included."""
import numpy as np
import pytest
import torch

import gpu_util as U
from paged_kv_cache_blocks_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def _ws(pa, b, grouped=False):
    w = b.workload
    f = pa.pa_decode_grouped_workspace_bytes if grouped else pa.pa_decode_workspace_bytes
    n = f(len(b.seq_lens), w.num_q_heads, w.head_dim, int(b.seq_lens.max()))
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("lens", [None, (0, 700, 5, 0, 2049, 3000, 1, 16)])
def test_reuse_plan_matches_full_call(pa, lens):
    """Layer 0 plans; layers 1 and 2 reuse the plan with other q / K / V and a
    NaN-filled output buffer: bit-identical to full calls, close to the oracle,
    zeros for empty sequences."""
    b = W.make_batch("llama8b", seed=3, num_layers=3, lens_override=list(lens) if lens else None)
    w = b.workload
    tab = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    msl = int(b.seq_lens.max())
    ws = _ws(pa, b)
    for layer in range(3):
        q, kc, vc, _, _ = U.device_inputs(b, layer)
        out = torch.full_like(q, float("nan"))
        pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl, out=out, workspace=ws,
                     reuse_plan=layer > 0)
        full = pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl)
        torch.cuda.synchronize()
        assert torch.equal(out, full), f"layer {layer}"
        got = out.double().cpu().numpy()
        empty = b.seq_lens == 0
        assert np.array_equal(got[empty], np.zeros_like(got[empty]))
        rows = np.flatnonzero(~empty)[:12]
        U.assert_close(got[rows], U.oracle_out(b, layer, rows=rows), f"reuse layer {layer}")


def test_reuse_plan_grouped_and_fp8(pa):
    """pa_decode_grouped and pa_decode_fp8 with a reused plan are bit-identical
    to their full calls."""
    b = U.batch("fullstep", num_layers=2)
    w = b.workload
    tab = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    goff, gpre = (torch.from_numpy(x).cuda() for x in b.group_arrays())
    msl = int(b.seq_lens.max())
    ws = _ws(pa, b, grouped=True)
    outs = []
    for layer in range(2):
        q, kc, vc, _, _ = U.device_inputs(b, layer)
        o = pa.pa_decode_grouped(q, kc, vc, tab, sl, w.scale, goff, gpre, max_seq_len=msl,
                                 workspace=ws, reuse_plan=layer > 0)
        outs.append(o.clone())
    for layer in range(2):
        q, kc, vc, _, _ = U.device_inputs(b, layer)
        full = pa.pa_decode_grouped(q, kc, vc, tab, sl, w.scale, goff, gpre, max_seq_len=msl)
        torch.cuda.synchronize()
        assert torch.equal(outs[layer], full), f"grouped layer {layer}"
    # FP8: a plan made by the 16-bit decode is the same plan
    b8 = U.batch("llama8b")
    q, kc, vc, tab, sl = U.device_inputs(b8)
    ks = torch.full((8,), 0.03, device="cuda")
    k8 = (kc.float() / 0.03).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (vc.float() / 0.03).to(torch.float8_e4m3fn).view(torch.uint8).transpose(2, 3).contiguous()
    ws8 = _ws(pa, b8)
    pa.pa_decode(q, kc, vc, tab, sl, b8.workload.scale, workspace=ws8)
    reused = pa.pa_decode_fp8(q, k8, v8, ks, ks, tab, sl, b8.workload.scale, workspace=ws8, reuse_plan=True)
    full = pa.pa_decode_fp8(q, k8, v8, ks, ks, tab, sl, b8.workload.scale)
    torch.cuda.synchronize()
    assert torch.equal(reused, full)
