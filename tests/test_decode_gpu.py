"""pa_decode on the GPU against the fp64 oracle, through the C ABI.

Every workload of the workload table is covered on every output row, at
full size and in the launch configuration the bench times (the 70B-shaped
batch of 256 sequences, two layers of the 32-layer shared-prefix step), with
both math variants.  Pools are NaN-poisoned wherever no token lives, so a
stray read shows up as a non-finite output."""
import numpy as np
import pytest
import torch

import gpu_util as U
from paged_kv_cache_blocks_gb300 import workloads as W

pytestmark = pytest.mark.gpu
VARIANTS = [1, 2]   # 1 = CUDA-core FMA, 2 = tensor-core mma


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def run(pa, b, layer=0, variant=0, **kw):
    q, kc, vc, tab, lens = U.device_inputs(b, layer)
    out = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale, variant=variant, **kw)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "llama8b", "long"])
def test_full_parity(pa, name, variant):
    b = U.batch(name)
    got = run(pa, b, variant=variant)
    U.assert_close(got, U.oracle_out(b), f"{name} v{variant}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_llama70b_mixed_all_rows(pa, variant):
    """The 70B-shaped mixed batch at full size (230 short and 26 long
    sequences, 918k tokens): every output row against the oracle."""
    b = U.batch("llama70b")
    got = run(pa, b, variant=variant)
    U.assert_close(got, U.oracle_out_cached("llama70b"), f"llama70b v{variant}")


def test_fullstep_two_layers_write_then_decode(pa):
    """Shared-prefix batch (4 groups x 32 sequences on one 1024-token prefix):
    cache write of the new token, then decode, per layer; every row."""
    b = U.batch("fullstep", num_layers=2)
    w = b.workload
    slots = torch.from_numpy(b.slot_mapping).cuda()
    tab = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    for layer in range(2):
        Lr = b.layers[layer]
        kc, vc = U.to_dev(Lr.k_cache, w.dtype).clone(), U.to_dev(Lr.v_cache, w.dtype).clone()
        pa.pa_cache_write(U.to_dev(Lr.new_k, w.dtype), U.to_dev(Lr.new_v, w.dtype), slots, kc, vc)
        out = pa.pa_decode(U.to_dev(Lr.q, w.dtype), kc, vc, tab, lens, w.scale)
        got = out.double().cpu().numpy()
        U.assert_close(got, U.oracle_out_cached("fullstep", layer, num_layers=2),
                       f"fullstep layer {layer}")


@pytest.mark.parametrize("name", ["tiny", "llama8b"])
def test_relabelled_blocks_give_identical_output(pa, name):
    b = U.batch(name)
    a = run(pa, b)
    r = W.relabel_blocks(b, 7)
    assert np.array_equal(a, run(pa, r))


@pytest.mark.parametrize("name", ["long", "llama70b"])
def test_repeated_calls_are_bit_identical(pa, name):
    """Work is handed out dynamically; the result must not depend on it."""
    b = U.batch(name)
    a = run(pa, b)
    for _ in range(2):
        assert np.array_equal(a, run(pa, b))


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1023, 1024, 1025, 1537, 2048, 3]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "llama70b", "llama8b"])
def test_edge_lengths(pa, name, variant):
    b = U.batch(name, seed=5, lens=tuple(EDGE_LENS))
    U.assert_close(run(pa, b, variant=variant), U.oracle_out(b), f"edges {name} v{variant}")


def test_2048_token_partitions_edges(pa):
    """Enough long sequences that the prep kernel picks 2048-token
    partitions; lengths around its multiples and tiny ones beside them."""
    lens = (32768,) * 20 + (2047, 2048, 2049, 4095, 4096, 4097, 1, 17, 1000, 6001)
    b = U.batch("llama70b", seed=8, lens=lens)
    q, kc, vc, tab, lens_d = U.device_inputs(b)
    ws = torch.empty(pa.pa_decode_workspace_bytes(len(lens), q.shape[1], q.shape[2],
                                                  b.block_tables.shape[1] * 16),
                     dtype=torch.uint8, device="cuda")
    for variant in (1, 2):
        out = pa.pa_decode(q, kc, vc, tab, lens_d, b.workload.scale, workspace=ws, variant=variant)
        torch.cuda.synchronize()
        assert int(ws[24:28].view(torch.int32).item()) == 2048
        got = out.double().cpu().numpy()
        rows = [0, 19] + list(range(20, len(lens)))
        U.assert_close(got[rows], U.oracle_out(b, rows=rows), f"2048-token partitions v{variant}")


def test_empty_sequences_give_zeros(pa):
    b = U.batch("llama8b", seed=6, lens=(0, 5, 0, 600))
    got = run(pa, b)
    assert np.array_equal(got[[0, 2]], np.zeros_like(got[[0, 2]]))
    U.assert_close(got[[1, 3]], U.oracle_out(b, rows=[1, 3]), "empty")


def test_device_error_flags_without_fault(pa):
    """A length past max_seq_len is clamped and flagged; a block id outside
    the pool reads zeros and is flagged; the other sequences stay right."""
    b = U.batch("llama8b", seed=7, lens=(40, 100, 60))
    q, kc, vc, tab, lens = U.device_inputs(b)
    ws = torch.empty(pa.pa_decode_workspace_bytes(3, q.shape[1], q.shape[2], 64),
                     dtype=torch.uint8, device="cuda")
    out = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale, max_seq_len=64, workspace=ws)
    bits = pa.pa_decode_check(ws)
    assert bits & pa.PA_DEVERR_SEQ_LEN
    got = out.double().cpu().numpy()
    U.assert_close(got[[0, 2]], U.oracle_out(b, rows=[0, 2]), "clamped neighbour")
    tab2 = tab.clone()
    tab2[1, 2] = b.num_blocks + 5
    out = pa.pa_decode(q, kc, vc, tab2, lens, b.workload.scale, workspace=ws)
    assert pa.pa_decode_check(ws) & pa.PA_DEVERR_BLOCK_ID
    got = out.double().cpu().numpy()
    U.assert_close(got[[0, 2]], U.oracle_out(b, rows=[0, 2]), "bad-id neighbour")
    out = pa.pa_decode(q, kc, vc, tab, lens, b.workload.scale, workspace=ws)
    assert pa.pa_decode_check(ws) == 0


def test_variants_agree_closely(pa):
    b = U.batch("llama8b")
    a, c = run(pa, b, variant=1), run(pa, b, variant=2)
    assert np.max(np.abs(a - c)) <= 1e-2


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("seed", range(3))
def test_random_batches(pa, seed, variant):
    """Seeded random batches mixing one-token, short and long sequences
    (1..12000 tokens) on the Llama-3-70B and -8B head layouts: every output
    row against the oracle."""
    rng = np.random.default_rng(2000 + seed)
    B = int(rng.integers(1, 97))
    kind = rng.integers(0, 10, B)
    lens = np.where(kind == 0, rng.integers(1, 17, B),
                    np.where(kind < 8, rng.integers(17, 2049, B), rng.integers(2049, 12001, B)))
    name = "llama70b" if seed % 2 == 0 else "llama8b"
    b = U.batch(name, seed=30 + seed, lens=tuple(int(x) for x in lens))
    got = run(pa, b, variant=variant)
    U.assert_close(got, U.oracle_out(b), f"random decode batch {seed} v{variant}")


def _ulp(ref, dtype):
    """One unit in the last place of the element type at |ref|."""
    return 2.0 * U.half_ulp(ref, dtype)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["llama8b", "tiny", "llama70b"])
def test_split_and_unsplit_agree(pa, name, variant):
    """Split-K on vs off: sequences of up to 2048 tokens decoded as one
    partition (the attention kernel writes the output itself) and as 512-token
    partitions whose partial results the merge kernel combines; longer
    sequences compare 512- against 2048-token partitions.

    The two differ by the rounding of each output (one unit in the last
    place between them) plus what the per-partition arithmetic rounds
    differently: with the weights P kept in fp32 (variant 1) only the fp32
    summation order, bounded here by 1e-5 x sum_t p_t |v_t| / sum_t p_t; on
    the tensor cores (variant 2) P enters the PV product in the element type,
    rounded against each partition's own running maximum, so each weight
    carries up to one unit roundoff u (2^-8 bf16, 2^-11 fp16) on either side:
    2u x sum_t p_t |v_t| / sum_t p_t.  The weighted |v| comes from the oracle
    (decode over |V|)."""
    lens = (2048, 2047, 1537, 1025, 1024, 600, 513, 512, 100, 1, 9000, 6145)
    b = U.batch(name, seed=9, lens=lens)
    w = b.workload
    q, kc, vc, tab, sl = U.device_inputs(b)
    ws = torch.empty(pa.pa_decode_workspace_bytes(len(lens), w.num_q_heads, w.head_dim, 9000),
                     dtype=torch.uint8, device="cuda")
    outs = {}
    for pt in (2048, 512):
        outs[pt] = pa.pa_decode(q, kc, vc, tab, sl, w.scale, max_seq_len=9000, workspace=ws,
                                partition_tokens=pt, variant=variant).double().cpu().numpy()
        assert int(ws[24:28].view(torch.int32).item()) == pt
        assert pa.pa_decode_check(ws) == 0
    a, c = outs[2048], outs[512]
    pk, pv = W.place_new_tokens(b, 0)
    pk, pv = pk.numpy().view(np.uint16), pv.numpy().view(np.uint16)
    weighted_abs_v = U.oracle_out(b, pools=(pk, pv & np.uint16(0x7FFF)))
    u = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}[w.dtype]
    rel = 1e-5 if variant == 1 else 2 * u
    bound = _ulp(np.maximum(np.abs(a), np.abs(c)), w.dtype) + rel * weighted_abs_v
    excess = np.abs(a - c) - bound
    assert excess.max() <= 0, (variant, float(np.abs(a - c).max()), float(excess.max()))
    ref = U.oracle_out(b)
    U.assert_close(a, ref, f"{name} one partition v{variant}")
    U.assert_close(c, ref, f"{name} 512-token partitions v{variant}")
