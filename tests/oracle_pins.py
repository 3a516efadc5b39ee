"""Pins that hold the oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (the default
build, or the variant passed as ``handle``) disagrees with what the pages or
the mathematics fix:

* worked numbers printed on the pages (tests/golden/*.json, each cited);
* library routines the definition reduces to (numpy / torch float decoding,
  ``torch.nn.functional.scaled_dot_product_attention`` in fp64 with the KV
  heads repeated for grouped-query attention);
* closed forms (one token, constant values, identical keys, one dominant key);
* invariants (the gather returns the contiguous source exactly; relabelling
  the physical blocks leaves the output bit-identical; a query never sees a
  token after its own position).

test_oracle.py runs every pin on the oracle; test_oracle_mutants.py plants
mistakes in copies of the oracle's source and checks that some pin fails.
"""
import json
import os

import numpy as np
import torch
import torch.nn.functional as F

from paged_kv_cache_blocks_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lib_f64(bits, dtype):
    """fp64 values of 16-bit patterns via numpy (fp16) / torch (bf16)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def sdpa_reference(batch, layer=0):
    """Per-sequence attention by the library routine, fp64, GQA by repeat."""
    w = batch.workload
    G = w.group_size
    q = lib_f64(batch.layers[layer].q.numpy().view(np.uint16), w.dtype)
    out = np.zeros((len(batch.seq_lens), w.num_q_heads, w.head_dim))
    for b, L in enumerate(batch.seq_lens):
        if L == 0:
            continue
        kb, vb = batch.contiguous_kv(layer, b)
        K = torch.from_numpy(lib_f64(kb, w.dtype)).permute(1, 0, 2)   # [Hkv, L, D]
        V = torch.from_numpy(lib_f64(vb, w.dtype)).permute(1, 0, 2)
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        qb = torch.from_numpy(q[b]).unsqueeze(1)                       # [Hq, 1, D]
        o = F.scaled_dot_product_attention(qb, K, V, scale=w.scale)
        out[b] = o[:, 0, :].numpy()
    return out


def small_batches():
    """Batches the oracle and the pins finish quickly on (several shapes)."""
    return [
        W.make_batch("tiny", seed=0, keep_contig=True),
        W.make_batch("llama8b", seed=1, keep_contig=True, lens_override=[5, 16, 31, 200, 1]),
        W.make_batch("llama70b", seed=2, keep_contig=True, lens_override=[48, 3, 130]),
        # three sequences sharing a 32-token prefix (one of them holds only the prefix)
        W.make_batch("llama8b", seed=3, keep_contig=True, lens_override=[40, 33, 32, 100, 5],
                     groups=[(3, 32), (1, 16), (1, 0)]),
    ]


def _decode(oracle, batch, handle, layer=0, pools=None):
    w = batch.workload
    q, _, _, _, _ = batch.np_layer(layer)
    if pools is None:
        kc, vc = W.place_new_tokens(batch, layer)
    else:
        kc, vc = pools
    return oracle.decode(q, kc.numpy().view(np.uint16), vc.numpy().view(np.uint16),
                         batch.block_tables, batch.seq_lens, w.scale, w.dtype, handle=handle)


# ----------------------------------------------------------------------------------

def pin_kv_bytes(oracle, handle=None):
    g = json.load(open(os.path.join(GOLD, "kv_bytes.json")))
    for c in g["per_token"]:
        assert oracle.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["bytes"]) \
            == c["expect"], c["cite"]
    for c in g["per_context"]:
        tot = oracle.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["bytes"]) \
            * c["tokens"]
        assert tot == c["expect_gib"] * 2 ** 30, c["cite"]


def pin_bits(oracle, handle=None):
    bits = np.arange(65536, dtype=np.uint16)
    for dt in ("f16", "bf16"):
        got = oracle.bits_to_double(bits, dt, handle=handle)
        ref = lib_f64(bits, dt)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan), dt
        assert np.array_equal(got[~nan], ref[~nan]), dt
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), dt


def pin_cache_write_golden(oracle, handle=None):
    g = json.load(open(os.path.join(GOLD, "cache_write_example.json")))
    bs, nb, H, D = g["block_size"], g["num_blocks"], g["num_kv_heads"], g["head_dim"]
    # small integers as fp16 patterns, so any misplaced copy is visible
    f = lambda x: np.asarray(x, np.float16).view(np.uint16)
    k, v = f(g["k"]), f(g["v"])
    kc0 = np.full((nb, H, bs, D), 0xFFFF, np.uint16)
    vc0 = kc0.copy()
    kc, vc, bad = oracle.cache_write(k, v, np.asarray(g["slots"], np.int64), kc0, vc0, bs,
                                     handle=handle)
    assert bad == g["expect_out_of_range"]
    ek, ev = kc0.copy(), vc0.copy()
    for e in g["expect_written"]:
        ek[e["block"], e["head"], e["row"]] = f(e["k"])
        ev[e["block"], e["head"], e["row"]] = f(e["v"])
    assert np.array_equal(kc, ek), g["cite"]
    assert np.array_equal(vc, ev), g["cite"]


def pin_copy_blocks_golden(oracle, handle=None):
    g = json.load(open(os.path.join(GOLD, "copy_blocks_example.json")))
    nb, H, D = g["num_blocks"], g["num_kv_heads"], g["head_dim"]
    b, h, r, d = np.meshgrid(np.arange(nb), np.arange(H), np.arange(16), np.arange(D), indexing="ij")
    vals = (1000 * b + 100 * h + 10 * (r % 10) + d).astype(np.float16).view(np.uint16)
    kc, vc = vals.copy(), (vals + 1).astype(np.uint16)
    k2, v2, skipped = oracle.copy_blocks(kc, vc, g["src"], g["dst"],
                                         handle=handle)
    assert skipped == g["expect_skipped"], g["cite"]
    for blk, srcb in enumerate(g["expect_block_source"]):
        assert np.array_equal(k2[blk], kc[srcb]), (blk, g["cite"])
        assert np.array_equal(v2[blk], vc[srcb]), (blk, g["cite"])


def pin_e4m3_codes(oracle, handle=None):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_double(codes, handle=handle)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    # rounding: every float in [-464, 464] to its nearest code, ties to even,
    # like torch; beyond that the code saturates to +-448 (torch gives NaN)
    rng = np.random.default_rng(3)
    vals = ref[~nan]
    mids = (np.sort(vals)[1:] + np.sort(vals)[:-1]) / 2
    x = np.concatenate([vals, mids, rng.uniform(-464, 464, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 1e-2, 5000), [464.0, -464.0]]).astype(np.float32)
    x = x[np.abs(x) <= 464]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.float_to_e4m3(x, handle=handle)
    assert np.array_equal(got, want)
    sat = oracle.float_to_e4m3(np.array([470.0, 1e9, -500.0, np.nan], np.float32), handle=handle)
    assert sat.tolist() == [0x7E, 0x7E, 0xFE, 0x7F]


def pin_cache_write_fp8_golden(oracle, handle=None):
    g = json.load(open(os.path.join(GOLD, "cache_write_fp8_example.json")))
    nb, D = g["num_blocks"], g["head_dim"]
    f = lambda x: torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)
    k8 = np.full((nb, 1, 16, D), 0xAA, np.uint8)
    v8 = np.full((nb, 1, D, 16), 0xAA, np.uint8)
    kc, vc, bad = oracle.cache_write_fp8(f(g["k"]), f(g["v"]), "bf16", np.array(g["slots"], np.int64),
                                         [g["k_scale"]], [g["v_scale"]], k8, v8, handle=handle)
    assert bad == 0
    ek, ev = k8.copy(), v8.copy()
    for e in g["expect_k"]:
        ek[e["block"], 0, e["row"], :] = e["codes"]
    for e in g["expect_v"]:
        ev[e["block"], 0, :, e["row"]] = e["codes"]
    assert np.array_equal(kc, ek), g["cite"]
    assert np.array_equal(vc, ev), g["cite"]


def pin_decode_fp8_reduces_to_decode(oracle, handle=None):
    """With power-of-two scales every dequantised value is exact in bf16, so
    FP8 decode must equal the (pinned) 16-bit decode on those values."""
    rng = np.random.default_rng(8)
    nb, H, D, G = 12, 2, 128, 4
    k8 = rng.integers(0, 256, (nb, H, 16, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, (nb, H, D, 16), dtype=np.uint8)
    for a in (k8, v8):   # no NaN codes; keep magnitudes moderate (exponent <= 8)
        a[(a & 0x7F) >= 0x78] &= 0x37
    ks, vs = np.array([0.25, 2.0], np.float32), np.array([0.5, 4.0], np.float32)
    lens = np.array([1, 16, 40, 130], np.int32)
    tab = np.array([[3, 0, 0, 0, 0, 0, 0, 0, 0], [7, 0, 0, 0, 0, 0, 0, 0, 0],
                    [1, 9, 4, 0, 0, 0, 0, 0, 0], [2, 5, 8, 10, 11, 0, 6, 1, 9]], np.int32)
    q = torch.randn((4, H * G, D), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    to_bf16 = lambda codes, sc: (torch.from_numpy(codes).view(torch.float8_e4m3fn).double()
                                 * torch.from_numpy(sc.astype(np.float64)).view(1, -1, 1, 1)) \
        .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kc = to_bf16(k8, ks)
    vc = to_bf16(np.ascontiguousarray(v8.transpose(0, 1, 3, 2)), vs)
    got = oracle.decode_fp8(q, k8, v8, ks, vs, tab, lens, 0.09, "bf16", handle=handle)
    ref = oracle.decode(q, kc, vc, tab, lens, 0.09, "bf16", handle=handle)
    assert np.array_equal(got, ref)


def pin_gather_is_contiguous_source(oracle, handle=None):
    for batch in small_batches():
        w = batch.workload
        kc, vc = W.place_new_tokens(batch, 0)
        kc, vc = kc.numpy().view(np.uint16), vc.numpy().view(np.uint16)
        for b, L in enumerate(batch.seq_lens):
            kb, vb = batch.contiguous_kv(0, b)
            for h in range(w.num_kv_heads):
                gk = oracle.gather(kc, w.dtype, batch.block_tables[b], int(L), h, handle=handle)
                gv = oracle.gather(vc, w.dtype, batch.block_tables[b], int(L), h, handle=handle)
                assert np.array_equal(gk, lib_f64(kb[:, h, :], w.dtype)), (w.name, b, h)
                assert np.array_equal(gv, lib_f64(vb[:, h, :], w.dtype)), (w.name, b, h)


def pin_matches_sdpa(oracle, handle=None):
    for batch in small_batches():
        got = _decode(oracle, batch, handle)
        ref = sdpa_reference(batch)
        err = np.max(np.abs(got - ref))
        assert err <= 1e-12, (batch.workload.name, err)


def pin_relabel_invariance(oracle, handle=None):
    for batch in small_batches():
        a = _decode(oracle, batch, handle)
        for s in (1, 2):
            r = W.relabel_blocks(batch, s)
            bb = _decode(oracle, r, handle)
            assert np.array_equal(a, bb), (batch.workload.name, s)


def _hand_pool(L, D, H, G, kvals, vvals, qvals, dtype="f16"):
    """One sequence stored in blocks laid out in reverse physical order."""
    bs = 16
    nblk = max(1, -(-L // bs))
    nb = nblk + 2
    table = np.arange(nb - 1, nb - 1 - nblk, -1, dtype=np.int32)[None, :]
    to_bits = (lambda x: np.asarray(x, np.float16).view(np.uint16)) if dtype == "f16" else \
        (lambda x: torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16)
         .numpy().view(np.uint16))
    kc = np.zeros((nb, H, bs, D), np.uint16)
    vc = np.zeros((nb, H, bs, D), np.uint16)
    for t in range(L):
        kc[table[0, t // bs], :, t % bs, :] = to_bits(kvals[t])
        vc[table[0, t // bs], :, t % bs, :] = to_bits(vvals[t])
    q = to_bits(qvals)[None]
    return q, kc, vc, table, np.asarray([L], np.int32)


def pin_closed_forms(oracle, handle=None):
    rng = np.random.default_rng(5)
    D, H, G = 8, 2, 2
    Hq = H * G
    scale = 0.25
    for dt in ("f16", "bf16"):
        # (1) one token: softmax of one score is 1, out = v
        kv = rng.integers(-8, 8, (1, H, D)).astype(np.float64) / 4
        vv = rng.integers(-8, 8, (1, H, D)).astype(np.float64) / 4
        qv = rng.integers(-8, 8, (Hq, D)).astype(np.float64) / 4
        q, kc, vc, t, ln = _hand_pool(1, D, H, G, kv, vv, qv, dt)
        o = oracle.decode(q, kc, vc, t, ln, scale, dt, handle=handle)
        for i in range(Hq):
            assert np.array_equal(o[0, i], vv[0, i // G]), ("one token", dt)
        # (2) constant values: out = that constant whatever the scores
        L = 37
        kv = rng.integers(-8, 8, (L, H, D)).astype(np.float64) / 4
        vv = np.full((L, H, D), 0.75)
        q, kc, vc, t, ln = _hand_pool(L, D, H, G, kv, vv, qv, dt)
        o = oracle.decode(q, kc, vc, t, ln, scale, dt, handle=handle)
        assert np.allclose(o, 0.75, rtol=0, atol=1e-14), ("constant V", dt)
        # (3) identical keys: uniform weights, out = mean of V over tokens
        kv = np.repeat(rng.integers(-8, 8, (1, H, D)).astype(np.float64) / 4, L, axis=0)
        vv = rng.integers(-8, 8, (L, H, D)).astype(np.float64) / 4
        q, kc, vc, t, ln = _hand_pool(L, D, H, G, kv, vv, qv, dt)
        o = oracle.decode(q, kc, vc, t, ln, scale, dt, handle=handle)
        for i in range(Hq):
            assert np.allclose(o[0, i], vv[:, i // G].mean(axis=0), rtol=0, atol=1e-13), \
                ("identical keys", dt)
        # (4) one key whose score leads all others by >= 50: out = its value
        j = 21
        kv = np.zeros((L, H, D))
        kv[j, :, 0] = 30.0
        qv = np.zeros((Hq, D))
        qv[:, 0] = 30.0   # score of key j: 900 * 0.25 = 225; others 0
        vv = rng.integers(-8, 8, (L, H, D)).astype(np.float64) / 4
        q, kc, vc, t, ln = _hand_pool(L, D, H, G, kv, vv, qv, dt)
        o = oracle.decode(q, kc, vc, t, ln, scale, dt, handle=handle)
        for i in range(Hq):
            assert np.allclose(o[0, i], vv[j, i // G], rtol=0, atol=1e-12), ("dominant key", dt)
    # (5) empty sequence: output defined as 0
    q, kc, vc, t, _ = _hand_pool(1, D, H, G, np.ones((1, H, D)), np.ones((1, H, D)),
                                 np.ones((Hq, D)))
    o = oracle.decode(q, kc, vc, t, np.asarray([0], np.int32), scale, "f16", handle=handle)
    assert np.array_equal(o, np.zeros_like(o))


# ---- multi-query (chunked prefill) attention -------------------------------------

def prefill_batches():
    """Multi-query batches with pieces in the middle of a prompt, whole
    prompts, single decode tokens, and pieces crossing block boundaries."""
    return [
        W.make_prefill_batch("tiny", seed=0, keep_contig=True, lens=[1, 17, 33, 100],
                             pieces=[1, 17, 9, 40]),
        W.make_prefill_batch("llama8b", seed=1, keep_contig=True, lens=[37, 300, 50, 16, 129],
                             pieces=[37, 1, 16, 3, 64]),
        W.make_prefill_batch("llama70b", seed=2, keep_contig=True, lens=[70, 5, 33],
                             pieces=[20, 5, 1]),
    ]


def sdpa_prefill_reference(pb, whole_prompt_causal=False):
    """Per-sequence attention by the library routine, fp64, GQA by repeat;
    query j of a piece of Qn tokens over L sees tokens t <= L - Qn + j (an
    explicit boolean mask, or is_causal=True when the piece is the whole
    prompt and ``whole_prompt_causal``)."""
    w = pb.workload
    G = w.group_size
    q = lib_f64(pb.q.numpy().view(np.uint16), w.dtype)
    out = np.zeros((pb.num_q_tokens, w.num_q_heads, w.head_dim))
    for b, L in enumerate(pb.seq_lens):
        L = int(L)
        n = int(pb.pieces[b])
        kb, vb = pb.contiguous_kv(b)
        K = torch.from_numpy(lib_f64(kb, w.dtype)).permute(1, 0, 2).repeat_interleave(G, dim=0)
        V = torch.from_numpy(lib_f64(vb, w.dtype)).permute(1, 0, 2).repeat_interleave(G, dim=0)
        q0 = int(pb.q_offsets[b])
        qb = torch.from_numpy(q[q0:q0 + n]).permute(1, 0, 2)            # [Hq, n, D]
        if whole_prompt_causal and n == L:
            o = F.scaled_dot_product_attention(qb, K, V, is_causal=True, scale=w.scale)
        else:
            mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
            o = F.scaled_dot_product_attention(qb, K, V, attn_mask=mask, scale=w.scale)
        out[q0:q0 + n] = o.permute(1, 0, 2).numpy()
    return out


def _prefill(oracle, pb, handle, rows=None, pools=None):
    w = pb.workload
    kc, vc = pb.placed_pools() if pools is None else pools
    return oracle.prefill(pb.q.numpy().view(np.uint16), kc.numpy().view(np.uint16),
                          vc.numpy().view(np.uint16), pb.block_tables, pb.seq_lens, pb.q_offsets,
                          w.scale, w.dtype, rows=rows, handle=handle)


def pin_prefill_matches_sdpa(oracle, handle=None):
    for pb in prefill_batches():
        got = _prefill(oracle, pb, handle)
        for causal in (False, True):
            err = np.max(np.abs(got - sdpa_prefill_reference(pb, causal)))
            assert err <= 1e-12, (pb.workload.name, causal, err)


def pin_prefill_causal_and_rows(oracle, handle=None):
    """A query never sees a later token: changing the K/V of a sequence's
    last token changes only that token's own query row.  Computing a subset
    of rows gives those rows bit-identically.  A piece of one token is the
    decode of that token (an independent SDPA pin holds the decode)."""
    pb = prefill_batches()[1]
    kc, vc = pb.placed_pools()
    full = _prefill(oracle, pb, handle, pools=(kc, vc))
    b = 4                                   # 129 tokens, piece of 64 (positions 65..128)
    last = int(pb.seq_lens[b]) - 1
    s = int(pb.block_tables[b, last // 16]) * 16 + last % 16
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[s // 16, :, s % 16, :] = pb.new_k[0]          # some other key
    vc2[s // 16, :, s % 16, :] = -vc2[s // 16, :, s % 16, :]
    mod = _prefill(oracle, pb, handle, pools=(kc2, vc2))
    q1 = int(pb.q_offsets[b + 1])
    same = np.ones(pb.num_q_tokens, bool)
    same[q1 - 1] = False
    assert np.array_equal(full[same], mod[same]), "a query saw a later token"
    assert not np.allclose(full[q1 - 1], mod[q1 - 1]), "the last query missed its own token"
    rows = np.array([q1 - 1, 0, 37, 38, 53, q1 - 64], np.int64)
    assert np.array_equal(_prefill(oracle, pb, handle, rows=rows), full[rows])
    # pieces of one token: the decode of each sequence's last token
    lens = np.array([5, 16, 200], np.int32)
    one = W.make_prefill_batch("llama8b", seed=4, lens=lens, pieces=[1, 1, 1])
    okc, ovc = one.placed_pools()
    dec = oracle.decode(one.q.numpy().view(np.uint16), okc.numpy().view(np.uint16),
                        ovc.numpy().view(np.uint16), one.block_tables, lens,
                        one.workload.scale, one.workload.dtype, handle=handle)
    assert np.array_equal(_prefill(oracle, one, handle), dec)


def pin_prefill_closed_forms(oracle, handle=None):
    """The first token of a prompt sees only itself: out = its v.  Constant
    values give that constant for every query of every piece."""
    pb = prefill_batches()[0]                          # tiny: fp16, d 64, G 2
    w = pb.workload
    got = _prefill(oracle, pb, handle)
    for b in range(len(pb.seq_lens)):
        if pb.pieces[b] == pb.seq_lens[b]:             # a whole prompt: row 0 is position 0
            q0 = int(pb.q_offsets[b])
            _, vb = pb.contiguous_kv(b)
            v0 = lib_f64(vb[0], w.dtype)               # [Hkv, D]
            for i in range(w.num_q_heads):
                assert np.array_equal(got[q0, i], v0[i // w.group_size]), ("position 0", b, i)
    kc, vc = pb.placed_pools()
    vc = torch.full_like(vc, int(np.float16(-1.25).view(np.int16)))
    got = _prefill(oracle, pb, handle, pools=(kc, vc))
    assert np.allclose(got, -1.25, rtol=0, atol=1e-14), "constant V"


def pin_prefill_relabel_invariance(oracle, handle=None):
    pb = prefill_batches()[1]
    a = _prefill(oracle, pb, handle)
    kc, vc = pb.placed_pools()
    rng = np.random.default_rng(9)
    perm = rng.permutation(pb.num_blocks)                # old id -> new id
    inv = np.argsort(perm)
    kc2, vc2 = kc[torch.from_numpy(inv)], vc[torch.from_numpy(inv)]
    pb2 = W.PrefillBatch(**{**pb.__dict__, "block_tables": perm[pb.block_tables].astype(np.int32)})
    b = oracle.prefill(pb.q.numpy().view(np.uint16), kc2.numpy().view(np.uint16),
                       vc2.numpy().view(np.uint16), pb2.block_tables, pb.seq_lens, pb.q_offsets,
                       pb.workload.scale, pb.workload.dtype, handle=handle)
    assert np.array_equal(a, b)


# ---- the dense form of the prefill oracle (matrix products as a step) ---------------

def _prefill_dense(oracle, pb, handle, rows=None, pools=None):
    w = pb.workload
    kc, vc = pb.placed_pools() if pools is None else pools
    return oracle.prefill_dense(pb.q.numpy().view(np.uint16), kc.numpy().view(np.uint16),
                                vc.numpy().view(np.uint16), pb.block_tables, pb.seq_lens,
                                pb.q_offsets, w.scale, w.dtype, rows=rows, handle=handle)


def pin_prefill_dense_matches_sdpa(oracle, handle=None):
    """The library routine on every row of the small batches, both mask forms."""
    for pb in prefill_batches():
        got = _prefill_dense(oracle, pb, handle)
        for causal in (False, True):
            err = np.max(np.abs(got - sdpa_prefill_reference(pb, causal)))
            assert err <= 1e-12, ("dense", pb.workload.name, causal, err)


def pin_prefill_dense_matches_loop_form(oracle, handle=None):
    """The scalar-loop prefill oracle (itself pinned to the library routine,
    causality, closed forms and relabelling) on the small batches and on
    rows across the first piece of the 30,000-token chunked workload (a piece
    of 3,750 tokens, 64 query heads, several row groups), to 1e-12."""
    for pb in prefill_batches():
        err = np.max(np.abs(_prefill_dense(oracle, pb, handle) - _prefill(oracle, pb, handle)))
        assert err <= 1e-12, ("dense vs loop", pb.workload.name, err)
    pb = W.make_prefill_batch("chunked", seed=0, iteration=1)
    rows = np.array([0, 1, 255, 256, 257, 1000, 1875, 3000, 3749, 3750, 3769], np.int64)
    kc, vc = pb.placed_pools()
    err = np.max(np.abs(_prefill_dense(oracle, pb, handle, rows=rows, pools=(kc, vc))
                        - _prefill(oracle, pb, handle, rows=rows, pools=(kc, vc))))
    assert err <= 1e-12, ("dense vs loop, chunked rows", err)


def pin_prefill_dense_causal_and_closed_forms(oracle, handle=None):
    """A query never sees a later token (only the last row changes when the
    last token's K/V change); position 0 of a whole prompt gives its own v
    exactly; constant V gives the constant; relabelling the physical blocks
    gives bit-identical output; a subset of rows gives those rows."""
    pb = prefill_batches()[1]
    kc, vc = pb.placed_pools()
    full = _prefill_dense(oracle, pb, handle, pools=(kc, vc))
    b = 4
    last = int(pb.seq_lens[b]) - 1
    s = int(pb.block_tables[b, last // 16]) * 16 + last % 16
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[s // 16, :, s % 16, :] = pb.new_k[0]
    vc2[s // 16, :, s % 16, :] = -vc2[s // 16, :, s % 16, :]
    mod = _prefill_dense(oracle, pb, handle, pools=(kc2, vc2))
    q1 = int(pb.q_offsets[b + 1])
    same = np.ones(pb.num_q_tokens, bool)
    same[q1 - 1] = False
    assert np.max(np.abs(full[same] - mod[same])) <= 1e-15, "a query saw a later token"
    assert not np.allclose(full[q1 - 1], mod[q1 - 1]), "the last query missed its own token"
    rows = np.array([q1 - 1, 0, 37, 38, 53, q1 - 64], np.int64)
    assert np.max(np.abs(_prefill_dense(oracle, pb, handle, rows=rows) - full[rows])) <= 1e-14
    perm = np.random.default_rng(9).permutation(pb.num_blocks)
    inv = torch.from_numpy(np.argsort(perm))
    pb2 = W.PrefillBatch(**{**pb.__dict__, "block_tables": perm[pb.block_tables].astype(np.int32)})
    assert np.array_equal(_prefill_dense(oracle, pb2, handle, pools=(kc[inv], vc[inv])), full)
    tb = prefill_batches()[0]                          # tiny: fp16, d 64, G 2
    w = tb.workload
    got = _prefill_dense(oracle, tb, handle)
    for bb in range(len(tb.seq_lens)):
        if tb.pieces[bb] == tb.seq_lens[bb]:
            q0 = int(tb.q_offsets[bb])
            v0 = lib_f64(tb.contiguous_kv(bb)[1][0], w.dtype)
            for i in range(w.num_q_heads):
                assert np.array_equal(got[q0, i], v0[i // w.group_size]), ("dense position 0", bb, i)
    tkc, tvc = tb.placed_pools()
    tvc = torch.full_like(tvc, int(np.float16(-1.25).view(np.int16)))
    got = _prefill_dense(oracle, tb, handle, pools=(tkc, tvc))
    assert np.allclose(got, -1.25, rtol=0, atol=1e-14), "dense constant V"


DENSE_PINS = [pin_prefill_dense_matches_sdpa, pin_prefill_dense_matches_loop_form,
              pin_prefill_dense_causal_and_closed_forms]

ALL_PINS = [pin_kv_bytes, pin_bits, pin_cache_write_golden, pin_copy_blocks_golden,
            pin_e4m3_codes, pin_cache_write_fp8_golden, pin_decode_fp8_reduces_to_decode,
            pin_gather_is_contiguous_source,
            pin_matches_sdpa, pin_relabel_invariance, pin_closed_forms,
            pin_prefill_matches_sdpa, pin_prefill_causal_and_rows, pin_prefill_closed_forms,
            pin_prefill_relabel_invariance] + DENSE_PINS
