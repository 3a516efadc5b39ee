"""Multi-query paged attention (chunked prefill) on the GPU against the fp64
oracle: pa_cache_write puts each piece's K/V into the pool, then pa_prefill
attends causally; the oracle computes the same rows from the same pool."""
import numpy as np
import pytest
import torch

import gpu_util as U
import oracle
from paged_kv_cache_blocks_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run(pa, pb, rows=None, pools=None, tables=None, write=True, variant=0):
    """GPU output (all rows) and the oracle's rows of one multi-query batch
    (variant: 0 auto, 2 mma.sync, 3 tcgen05)."""
    w = pb.workload
    dt = U.TORCH_DT[w.dtype]
    if pools is None:
        kc, vc = U.to_dev(pb.k_cache, w.dtype), U.to_dev(pb.v_cache, w.dtype)
        if write:
            pa.pa_cache_write(U.to_dev(pb.new_k, w.dtype), U.to_dev(pb.new_v, w.dtype),
                              torch.from_numpy(pb.slot_mapping).cuda(), kc, vc)
        else:
            pk, pv = pb.placed_pools()
            kc, vc = U.to_dev(pk, w.dtype), U.to_dev(pv, w.dtype)
    else:
        kc, vc = pools
    tab = pb.block_tables if tables is None else tables
    ws = torch.empty(max(pa.pa_prefill_workspace_bytes(len(pb.seq_lens), pb.num_q_tokens,
                                                       w.num_q_heads, w.num_kv_heads), 256),
                     dtype=torch.uint8, device="cuda")
    out = pa.pa_prefill(U.to_dev(pb.q, w.dtype), kc, vc, torch.from_numpy(tab).cuda(),
                        torch.from_numpy(pb.seq_lens).cuda(), torch.from_numpy(pb.q_offsets).cuda(),
                        w.scale, workspace=ws, variant=variant)
    torch.cuda.synchronize()
    assert pa.pa_decode_check(ws) == 0
    got = out.double().cpu().numpy()
    ref = oracle.prefill(_u16(pb.q), _u16(kc), _u16(vc), tab, pb.seq_lens, pb.q_offsets, w.scale,
                         w.dtype, rows=rows)
    return (got if rows is None else got[rows]), ref, out


SMALL = [
    # (workload, lens, pieces): whole prompts, pieces mid-prompt, decode tokens,
    # pieces crossing blocks and spanning several 128-row tiles
    ("tiny", [1, 17, 33, 100], [1, 17, 9, 40]),
    ("llama8b", [37, 300, 50, 16, 129, 700], [37, 1, 16, 3, 64, 300]),
    ("llama70b", [70, 5, 33, 600, 1000], [20, 5, 1, 200, 17]),
]


CASES = [(n, l, p, v) for n, l, p in SMALL for v in ((2,) if n == "tiny" else (2, 3))]


@pytest.mark.parametrize("name,lens,pieces,variant", CASES,
                         ids=[f"{c[0]}-{'tc' if c[3] == 3 else 'mma'}" for c in CASES])
def test_prefill_small_all_rows(pa, name, lens, pieces, variant):
    pb = W.make_prefill_batch(name, seed=3, lens=lens, pieces=pieces)
    got, ref, _ = run(pa, pb, variant=variant)
    U.assert_close_rounded(got, ref, pb.workload.dtype, f"prefill {name} variant {variant}")


@pytest.mark.parametrize("variant", [2, 3])
def test_prefill_fp16_g4_both_variants(pa, variant):
    """fp16 operands on the tensor cores (the tcgen05 kind::f16 with fp16 A/B)."""
    import dataclasses
    W.WORKLOADS["f16g4"] = dataclasses.replace(W.WORKLOADS["llama8b"], name="f16g4", dtype="f16")
    W._SEED_SALT["f16g4"] = 78
    try:
        pb = W.make_prefill_batch("f16g4", seed=2, lens=[300, 47, 1000], pieces=[150, 47, 3])
        got, ref, _ = run(pa, pb, variant=variant)
        U.assert_close_rounded(got, ref, "f16", f"prefill fp16 variant {variant}")
    finally:
        del W.WORKLOADS["f16g4"], W._SEED_SALT["f16g4"]


def test_prefill_one_query_head_per_kv_head(pa):
    """G = 1 (tiles of 128 query tokens), fp16, head_dim 64."""
    lens, pieces = [300, 129, 64, 1], [260, 129, 1, 1]
    w = W.WORKLOADS["tiny"]
    import dataclasses
    W.WORKLOADS["g1"] = dataclasses.replace(w, name="g1", num_q_heads=2, num_kv_heads=2)
    W._SEED_SALT["g1"] = 77
    try:
        pb = W.make_prefill_batch("g1", seed=1, lens=lens, pieces=pieces)
        got, ref, _ = run(pa, pb)
        U.assert_close_rounded(got, ref, "f16", "prefill G=1")
    finally:
        del W.WORKLOADS["g1"], W._SEED_SALT["g1"]


_CHUNKED_REF = {}


def chunked_reference(pb, iteration):
    """Every output row of one iteration of the chunked workload from the
    oracle's dense form (the loop form would take tens of minutes on the
    last pieces), computed once per process."""
    if iteration not in _CHUNKED_REF:
        w = pb.workload
        kc, vc = pb.placed_pools()
        _CHUNKED_REF[iteration] = oracle.prefill_dense(
            pb.q.numpy().view(np.uint16), kc.numpy().view(np.uint16), vc.numpy().view(np.uint16),
            pb.block_tables, pb.seq_lens, pb.q_offsets, w.scale, w.dtype)
    return _CHUNKED_REF[iteration]


@pytest.mark.parametrize("iteration,variant", [(1, 3), (8, 3), (8, 2)])
def test_prefill_chunked_workload_all_rows(pa, iteration, variant):
    """The full chunked workload (30000-token prompt, piece k of 8 -- 3,750
    query tokens over up to 30,000 keys -- plus 20 decode tokens), in the
    launch configuration the bench times: every output row against the
    oracle.  The pools the GPU cache write produced are byte-identical to the
    oracle's placement first."""
    pb = W.make_prefill_batch("chunked", seed=0, iteration=iteration)
    w = pb.workload
    kc, vc = U.to_dev(pb.k_cache, w.dtype), U.to_dev(pb.v_cache, w.dtype)
    pa.pa_cache_write(U.to_dev(pb.new_k, w.dtype), U.to_dev(pb.new_v, w.dtype),
                      torch.from_numpy(pb.slot_mapping).cuda(), kc, vc)
    pk, pv = pb.placed_pools()
    assert np.array_equal(_u16(kc), pk.numpy().view(np.uint16))
    assert np.array_equal(_u16(vc), pv.numpy().view(np.uint16))
    ws = torch.empty(pa.pa_prefill_workspace_bytes(len(pb.seq_lens), pb.num_q_tokens,
                                                   w.num_q_heads, w.num_kv_heads),
                     dtype=torch.uint8, device="cuda")
    out = pa.pa_prefill(U.to_dev(pb.q, w.dtype), kc, vc, torch.from_numpy(pb.block_tables).cuda(),
                        torch.from_numpy(pb.seq_lens).cuda(), torch.from_numpy(pb.q_offsets).cuda(),
                        w.scale, workspace=ws, variant=variant)
    torch.cuda.synchronize()
    assert pa.pa_decode_check(ws) == 0
    U.assert_close_rounded(out.double().cpu().numpy(), chunked_reference(pb, iteration), "bf16",
                           f"chunked iteration {iteration} variant {variant}")


def test_prefill_decode_tokens_match_pa_decode(pa):
    """Pieces of one token are decode steps: pa_prefill and pa_decode agree."""
    pb = W.make_prefill_batch("llama8b", seed=6, lens=[1, 16, 17, 511, 2000, 33],
                              pieces=[1] * 6)
    got, ref, out = run(pa, pb)
    U.assert_close_rounded(got, ref, "bf16", "decode-shaped prefill")
    kc, vc = pb.placed_pools()
    dec = pa.pa_decode(U.to_dev(pb.q, "bf16"), U.to_dev(kc, "bf16"), U.to_dev(vc, "bf16"),
                       torch.from_numpy(pb.block_tables).cuda(),
                       torch.from_numpy(pb.seq_lens).cuda(), pb.workload.scale)
    torch.cuda.synchronize()
    assert (out.double() - dec.double()).abs().max().item() <= 2e-2


@pytest.mark.parametrize("variant", [2, 3])
def test_prefill_deterministic_and_relabel_invariant(pa, variant):
    """Every row is summed in block order by one warp (mma.sync) or one
    thread and the tensor cores (tcgen05): repeated calls and a relabelling of
    the physical blocks give bit-identical outputs."""
    pb = W.make_prefill_batch("llama70b", seed=8, lens=[900, 40, 333], pieces=[400, 1, 100])
    _, _, a = run(pa, pb, rows=np.array([0], np.int64), write=False, variant=variant)
    _, _, b = run(pa, pb, rows=np.array([0], np.int64), write=False, variant=variant)
    assert torch.equal(a, b)
    pk, pv = pb.placed_pools()
    perm = np.random.default_rng(2).permutation(pb.num_blocks)
    inv = torch.from_numpy(np.argsort(perm))
    pools = (U.to_dev(pk[inv], "bf16"), U.to_dev(pv[inv], "bf16"))
    _, _, c = run(pa, pb, rows=np.array([0], np.int64), pools=pools,
                  tables=perm[pb.block_tables].astype(np.int32), variant=variant)
    assert torch.equal(a, c)


def test_prefill_flags_bad_input_without_faulting(pa):
    """A piece longer than its sequence and a block id outside the pool are
    flagged; the call completes."""
    pb = W.make_prefill_batch("llama8b", seed=9, lens=[40, 20], pieces=[10, 4])
    w = pb.workload
    kc, vc = pb.placed_pools()
    kc, vc = U.to_dev(kc, w.dtype), U.to_dev(vc, w.dtype)
    ws = torch.empty(pa.pa_prefill_workspace_bytes(2, pb.num_q_tokens, w.num_q_heads,
                                                   w.num_kv_heads), dtype=torch.uint8, device="cuda")
    q = U.to_dev(pb.q, w.dtype)
    tab = torch.from_numpy(pb.block_tables).cuda()
    bad_lens = torch.tensor([40, 3], dtype=torch.int32, device="cuda")     # piece of 4 > 3
    pa.pa_prefill(q, kc, vc, tab, bad_lens, torch.from_numpy(pb.q_offsets).cuda(), w.scale,
                  workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_decode_check(ws) & 1
    tab2 = tab.clone()
    tab2[0, 1] = pb.num_blocks + 5
    out = pa.pa_prefill(q, kc, vc, tab2, torch.from_numpy(pb.seq_lens).cuda(),
                        torch.from_numpy(pb.q_offsets).cuda(), w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_decode_check(ws) & 2
    # rows of the sequence with the good table are unaffected
    ref = oracle.prefill(_u16(pb.q), _u16(kc), _u16(vc), pb.block_tables, pb.seq_lens,
                         pb.q_offsets, w.scale, w.dtype)
    U.assert_close_rounded(out[10:].double().cpu().numpy(), ref[10:], "bf16",
                           "rows after a bad block id")


@pytest.mark.parametrize("variant", [2, 3])
@pytest.mark.parametrize("hq", [8, 16])
def test_prefill_head_dim_128_small_groups(pa, hq, variant):
    """G = 1 (Q box of 128 tokens x 1 head) and G = 2 (64 tokens x 2 heads) at
    head_dim 128, where the tcgen05 kernel applies."""
    import dataclasses
    name = f"g{hq // 8}d128"
    W.WORKLOADS[name] = dataclasses.replace(W.WORKLOADS["llama8b"], name=name, num_q_heads=hq)
    W._SEED_SALT[name] = 80 + hq
    try:
        pb = W.make_prefill_batch(name, seed=4, lens=[400, 129, 1000, 7], pieces=[300, 129, 2, 7])
        got, ref, _ = run(pa, pb, variant=variant)
        U.assert_close_rounded(got, ref, "bf16", f"prefill G={hq // 8} d128 variant {variant}")
    finally:
        del W.WORKLOADS[name], W._SEED_SALT[name]


@pytest.mark.parametrize("variant", [2, 3])
def test_prefill_empty_pieces_and_empty_sequences(pa, variant):
    """Sequences with no query token this iteration (empty pieces) or with no
    tokens at all, beside pieces of one token, of a few and of several tiles."""
    pb = W.make_prefill_batch("llama70b", seed=11, lens=[0, 5, 300, 17, 129, 16, 0],
                              pieces=[0, 0, 130, 17, 1, 16, 0])
    got, ref, _ = run(pa, pb, variant=variant)
    assert got.shape[0] == 164
    U.assert_close_rounded(got, ref, "bf16", f"empty pieces variant {variant}")


@pytest.mark.parametrize("variant", [2, 3])
def test_prefill_without_query_tokens_is_a_noop(pa, variant):
    """Every piece empty: the call returns at once with an empty output."""
    pb = W.make_prefill_batch("llama8b", seed=12, lens=[40, 0, 17], pieces=[0, 0, 0])
    w = pb.workload
    kc, vc = pb.placed_pools()
    out = pa.pa_prefill(U.to_dev(pb.q, w.dtype), U.to_dev(kc, w.dtype), U.to_dev(vc, w.dtype),
                        torch.from_numpy(pb.block_tables).cuda(), torch.from_numpy(pb.seq_lens).cuda(),
                        torch.from_numpy(pb.q_offsets).cuda(), w.scale, variant=variant)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, w.num_q_heads, w.head_dim)


def _random_shape(seed):
    """A seeded random batch shape: 1..10 sequences of 1..2000 tokens, pieces
    of 0..300 tokens (some of one token, some empty)."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 11))
    lens = rng.integers(1, 2001, B)
    pieces = np.minimum(lens, rng.integers(1, 301, B))
    kind = rng.integers(0, 4, B)
    pieces = np.where(kind == 0, 1, pieces)                 # decode tokens
    pieces = np.where((kind == 1) & (B > 1), 0, pieces)     # sequences idle this iteration
    return lens.tolist(), pieces.tolist()


@pytest.mark.parametrize("variant", [2, 3])
@pytest.mark.parametrize("seed", range(4))
def test_prefill_random_batches(pa, seed, variant):
    """Seeded random batches on the Llama-3-70B and -8B head layouts: every
    output row against the oracle."""
    name = "llama70b" if seed % 2 == 0 else "llama8b"
    lens, pieces = _random_shape(seed)
    pb = W.make_prefill_batch(name, seed=20 + seed, lens=lens, pieces=pieces)
    got, ref, _ = run(pa, pb, variant=variant)
    U.assert_close_rounded(got, ref, pb.workload.dtype, f"random batch {seed} variant {variant}")


@pytest.mark.parametrize("nseq", [4096, 4100])
def test_prefill_many_sequences(pa, nseq):
    """Thousands of sequences (decode tokens and short pieces): the prep kernel
    lists tiles from a shared-memory prefix sum up to 4096 sequences and per
    sequence beyond; both against the oracle on every row."""
    rng = np.random.default_rng(nseq)
    lens = rng.integers(1, 65, nseq)
    pieces = np.minimum(lens, np.where(rng.random(nseq) < 0.9, 1, rng.integers(1, 40, nseq)))
    pieces[rng.random(nseq) < 0.05] = 0
    pb = W.make_prefill_batch("llama8b", seed=40, lens=lens.tolist(), pieces=pieces.tolist())
    got, ref, _ = run(pa, pb, variant=3)
    U.assert_close_rounded(got, ref, "bf16", f"{nseq} sequences")
