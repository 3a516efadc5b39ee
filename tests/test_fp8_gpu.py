"""FP8 (E4M3) KV cache on the GPU: pa_cache_write_fp8 byte-identical to the
oracle's quantising scatter, pa_decode_fp8 against the oracle's fp64
attention over the same dequantised codes."""
import numpy as np
import pytest
import torch

import gpu_util as U
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def scales(H):
    ks = np.array([0.02 + 0.005 * h for h in range(H)], np.float32)
    vs = np.array([0.03 + 0.004 * h for h in range(H)], np.float32)
    return ks, vs


def quantise_pool(b, layer, ks, vs):
    """E4M3 codes of a batch's 16-bit pools (new tokens placed), K token-major,
    V dimension-major; NaN slots stay NaN codes.  Values stay far below 448."""
    kc, vc = U.device_inputs(b, layer)[1:3]
    kk = torch.from_numpy(1.0 / ks).cuda().view(1, -1, 1, 1)
    vv = torch.from_numpy(1.0 / vs).cuda().view(1, -1, 1, 1)
    k8 = (kc.float() * kk).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (vc.float() * vv).to(torch.float8_e4m3fn).view(torch.uint8).transpose(2, 3).contiguous()
    return k8, v8


def run_fp8(pa, b, ks, vs, rows=None):
    w = b.workload
    q, _, _, tab, lens = U.device_inputs(b)
    k8, v8 = quantise_pool(b, 0, ks, vs)
    out = pa.pa_decode_fp8(q, k8, v8, torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(), tab,
                           lens, w.scale)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    qn = b.layers[0].q.numpy().view(np.uint16)
    tb, ln = b.block_tables, b.seq_lens
    if rows is not None:
        qn, tb, ln, got = qn[rows], tb[rows], ln[rows], got[rows]
    ref = oracle.decode_fp8(qn, k8.cpu().numpy(), v8.cpu().numpy(), ks, vs, tb, ln, w.scale, w.dtype)
    return got, ref


@pytest.mark.parametrize("name", ["llama8b", "long"])
def test_decode_fp8_full(pa, name):
    b = U.batch(name)
    ks, vs = scales(b.workload.num_kv_heads)
    got, ref = run_fp8(pa, b, ks, vs)
    U.assert_close(got, ref, f"fp8 {name}")


def test_decode_fp8_llama70b_all_rows(pa):
    """The 70B-shaped mixed batch at full size: every output row."""
    b = U.batch("llama70b")
    ks, vs = scales(8)
    got, ref = run_fp8(pa, b, ks, vs)
    U.assert_close(got, ref, "fp8 llama70b")


@pytest.mark.parametrize("name", ["llama8b", "llama70b"])
def test_decode_fp8_edge_lengths(pa, name):
    lens = (1, 2, 15, 16, 17, 31, 33, 511, 512, 513, 1025, 3)
    b = U.batch(name, seed=5, lens=lens)
    ks, vs = scales(8)
    got, ref = run_fp8(pa, b, ks, vs)
    U.assert_close(got, ref, f"fp8 edges {name}")


def test_fp8_close_to_bf16(pa):
    """Quantisation error only: FP8 and bf16 decodes of the same batch agree to
    a few percent of the output scale."""
    b = U.batch("llama8b")
    ks, vs = scales(8)
    got, _ = run_fp8(pa, b, ks, vs)
    q, kc, vc, tab, lens = U.device_inputs(b)
    ref16 = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale).double().cpu().numpy()
    assert np.mean(np.abs(got - ref16)) < 0.02


def test_cache_write_fp8_bit_exact(pa):
    b = U.batch("llama70b")
    w = b.workload
    ks = np.array([0.37, 0.011, 1.7, 0.05, 0.123, 0.09, 3.3, 0.0007], np.float32)
    vs = np.array([0.21, 0.5, 0.013, 0.77, 0.031, 0.058, 1.01, 0.24], np.float32)
    rng = np.random.default_rng(2)
    T = 2000
    slots = rng.choice(4096 * 16, size=T, replace=False).astype(np.int64)
    slots[::9] = -1
    slots[4] = 4096 * 16 + 5                       # past the pool
    gen = torch.Generator().manual_seed(4)
    k = (torch.randn((T, 8, 128), generator=gen) * 3).to(torch.bfloat16)
    v = (torch.randn((T, 8, 128), generator=gen) * 3).to(torch.bfloat16)
    k[0, 0, :4] = torch.tensor([1e6, -1e6, float("nan"), 0.0])   # saturation, NaN, zero
    k8 = torch.full((4096, 8, 16, 128), 0x55, dtype=torch.uint8, device="cuda")
    v8 = torch.full((4096, 8, 128, 16), 0x55, dtype=torch.uint8, device="cuda")
    pa.pa_cache_write_fp8(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(),
                          torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(), k8, v8)
    torch.cuda.synchronize()
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    ok, ov, bad = oracle.cache_write_fp8(u16(k), u16(v), "bf16", slots, ks, vs,
                                         np.full((4096, 8, 16, 128), 0x55, np.uint8),
                                         np.full((4096, 8, 128, 16), 0x55, np.uint8))
    assert bad == 1
    assert np.array_equal(k8.cpu().numpy(), ok) and np.array_equal(v8.cpu().numpy(), ov)
    del w
