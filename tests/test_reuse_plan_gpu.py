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


def test_reuse_with_other_shapes_is_refused(pa):
    """A workspace planned for one batch refuses reuse with another batch's
    shapes (and after a prefill overwrote it): PA_ERR_INVALID on the host,
    nothing launched, the output buffer untouched."""
    a = W.make_batch("llama8b", seed=11, lens_override=[100, 700, 1500, 33])
    bb = W.make_batch("llama8b", seed=12, lens_override=[100, 700, 1500, 33, 9])
    w = a.workload
    ws = torch.empty(pa.pa_decode_workspace_bytes(5, w.num_q_heads, w.head_dim, 1500),
                     dtype=torch.uint8, device="cuda")
    q, kc, vc, tab, sl = U.device_inputs(a)
    pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=1500, workspace=ws)
    torch.cuda.synchronize()
    qb, kb, vb, tb, lb = U.device_inputs(bb)
    for args in ((qb, kb, vb, tb, lb, 1500),       # another batch size
                 (q, kc, vc, tab, sl, 1400)):       # another max_seq_len
        out = torch.full_like(args[0], float("nan"))
        with pytest.raises(pa.PaError) as e:
            pa.pa_decode(*args[:5], w.scale, max_seq_len=args[5], out=out, workspace=ws,
                         reuse_plan=True)
        assert e.value.code == pa.PA_ERR_INVALID
        torch.cuda.synchronize()
        assert torch.isnan(out).all()
    # same shapes as the planning call: accepted
    out = pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=1500, workspace=ws,
                       reuse_plan=True)
    torch.cuda.synchronize()
    assert pa.pa_decode_check(ws) == 0
    U.assert_close(out.double().cpu().numpy(), U.oracle_out(a), "reuse, same shapes")
    # a workspace no grouped call planned is refused to a grouped reuse
    with pytest.raises(pa.PaError) as e:
        goff = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
        gpre = torch.zeros(1, dtype=torch.int32, device="cuda")
        big = torch.empty(pa.pa_decode_grouped_workspace_bytes(4, w.num_q_heads, w.head_dim, 1500),
                          dtype=torch.uint8, device="cuda")
        pa.pa_decode_grouped(q, kc, vc, tab, sl, w.scale, goff, gpre, max_seq_len=1500,
                             workspace=big, reuse_plan=True)
    assert e.value.code == pa.PA_ERR_INVALID


def test_reuse_with_stale_lengths_is_flagged(pa):
    """Reuse with the planned shapes but other lengths: the plan is a valid
    plan of the workspace, so nothing leaves its buffers, and the lengths that
    differ from the plan's set PA_DEVERR_PLAN.  A planning call afterwards is
    clean and correct."""
    a = W.make_batch("llama8b", seed=13, lens_override=[300, 2000, 40, 1200])
    w = a.workload
    q, kc, vc, tab, sl = U.device_inputs(a)
    msl = 2000
    ws = torch.empty(pa.pa_decode_workspace_bytes(4, w.num_q_heads, w.head_dim, msl),
                     dtype=torch.uint8, device="cuda")
    pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl, workspace=ws)
    assert pa.pa_decode_check(ws) == 0
    shorter = (sl - 17).clamp(min=1)
    pa.pa_decode(q, kc, vc, tab, shorter, w.scale, max_seq_len=msl, workspace=ws, reuse_plan=True)
    assert pa.pa_decode_check(ws) & pa.PA_DEVERR_PLAN
    out = pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl, workspace=ws)
    assert pa.pa_decode_check(ws) == 0
    U.assert_close(out.double().cpu().numpy(), U.oracle_out(a), "after a stale reuse")


def _plan_words(B, msl):
    """int32 words of the workspace that hold the plan: header, partition
    records, per-sequence first partitions and merge records (the layout of
    the decode workspace: a 256-byte header, then 32-byte partition records
    for B x ceil(msl / 512) partitions, then 8 bytes and 32 bytes per
    sequence, each region starting on a 256-byte boundary)."""
    up = lambda x: (x + 255) // 256 * 256
    max_parts = B * -(-msl // 512)
    off_seq_first = up(256 + 32 * max_parts)
    off_split = up(off_seq_first + 8 * B)
    end = up(off_split + 32 * B)
    return end // 4


@pytest.mark.parametrize("mode", ["random", "random-valid-header", "perturbed", "negative-counter"])
def test_corrupted_plan_is_skipped_not_followed(pa, mode):
    """The plan lives in caller memory, so a reuse must not trust it: after a
    planning call the plan is overwritten (seeded: random words mixing small
    integers around the valid ranges, large and negative ones and zeros; or
    the true plan with words shifted by small amounts; or a work counter
    left negative) and reused.  The kernels' own bounds checks skip every
    record that does not fit the call's buffers and set PA_DEVERR_PLAN; the
    context stays usable and a planning call afterwards is correct."""
    a = W.make_batch("llama70b", seed=14, lens_override=[5000, 300, 17, 2100, 9000, 1])
    w = a.workload
    q, kc, vc, tab, sl = U.device_inputs(a)
    B, msl = 6, 9000
    ws = torch.empty(pa.pa_decode_workspace_bytes(B, w.num_q_heads, w.head_dim, msl),
                     dtype=torch.uint8, device="cuda")
    pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl, workspace=ws)
    torch.cuda.synchronize()
    nw = _plan_words(B, msl)
    plan = ws.view(torch.int32)[:nw].cpu()
    g = torch.Generator().manual_seed(500 + len(mode))
    n = nw
    kind = torch.randint(0, 4, (n,), generator=g)
    small = torch.randint(-3, 40, (n,), generator=g, dtype=torch.int32)
    near = torch.randint(0, 3000, (n,), generator=g, dtype=torch.int32)
    wide = torch.randint(-2**31, 2**31 - 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)
    if mode == "perturbed":
        shift = torch.randint(-40, 41, (n,), generator=g, dtype=torch.int32)
        words = torch.where(kind < 2, plan + shift, plan)
    elif mode == "negative-counter":
        words = plan.clone()
        words[3] = -5                  # the attention kernel's work counter
    else:
        words = torch.where(kind == 0, small, torch.where(kind == 1, near,
                            torch.where(kind == 2, wide, torch.zeros_like(small))))
        if mode == "random-valid-header":
            words[2], words[3], words[4], words[6] = 10 ** 6, 0, 5, 512
    words[0] = 0                      # error bits
    ws.view(torch.int32)[:nw].copy_(words.cuda())
    pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl, workspace=ws, reuse_plan=True)
    bits = pa.pa_decode_check(ws)
    assert not bits & pa.PA_DEVERR_TIMEOUT
    if mode != "perturbed":           # a shifted plan may still fit (then nothing is flagged)
        assert bits & pa.PA_DEVERR_PLAN
    out = pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=msl, workspace=ws)
    assert pa.pa_decode_check(ws) == 0
    U.assert_close(out.double().cpu().numpy(), U.oracle_out(a), f"after a corrupted plan ({mode})")
