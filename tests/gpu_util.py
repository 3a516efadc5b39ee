"""Helpers for the GPU parity tests: device copies of a workload batch, the
CUDA path through the C ABI, the oracle on the same inputs, comparisons."""
import functools

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_blocks_gb300 import workloads as W

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
# Tolerance on unit-scale inputs against the fp64 oracle (max and mean |error|
# over all compared outputs).
MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_blocks_gb300 import build, binding
    build.build()
    binding.lib()
    return binding


@functools.lru_cache(maxsize=4)
def batch(name, seed=0, num_layers=None, lens=None):
    return W.make_batch(name, seed=seed, num_layers=num_layers,
                        lens_override=list(lens) if lens is not None else None)


def to_dev(t, dtype):
    return t.to("cuda").view(TORCH_DT[dtype])


def device_inputs(b, layer=0, placed=True):
    """q, k_cache, v_cache (new tokens placed or not), tables, lens on the GPU."""
    w = b.workload
    Lr = b.layers[layer]
    if placed:
        kc, vc = W.place_new_tokens(b, layer)
    else:
        kc, vc = Lr.k_cache, Lr.v_cache
    return (to_dev(Lr.q, w.dtype), to_dev(kc, w.dtype), to_dev(vc, w.dtype),
            torch.from_numpy(b.block_tables).cuda(), torch.from_numpy(b.seq_lens).cuda())


def oracle_out(b, layer=0, rows=None, pools=None):
    """fp64 oracle outputs for `rows` (all when None) of one layer."""
    w = b.workload
    q, _, _, _, _ = b.np_layer(layer)
    if pools is None:
        kc, vc = W.place_new_tokens(b, layer)
        kc, vc = kc.numpy().view(np.uint16), vc.numpy().view(np.uint16)
    else:
        kc, vc = pools
    tab, lens = b.block_tables, b.seq_lens
    if rows is not None:
        rows = np.asarray(rows)
        q, tab, lens = q[rows], tab[rows], lens[rows]
    return oracle.decode(q, kc, vc, tab, lens, w.scale, w.dtype)


_ORACLE_CACHE = {}


def oracle_out_cached(name, layer=0, num_layers=None):
    """oracle_out of every row of a default workload batch, computed once per
    process (several tests compare the same full-size batch)."""
    key = (name, layer, num_layers)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle_out(batch(name, num_layers=num_layers), layer)
    return _ORACLE_CACHE[key]


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def half_ulp(ref, dtype):
    """Half a unit in the last place of the element type at |ref| (the
    rounding error of a correctly rounded output)."""
    mant = {"bf16": 8, "f16": 11}[dtype]          # significand bits, implicit one included
    a = np.maximum(np.abs(ref), {"bf16": 2.0 ** -126, "f16": 2.0 ** -14}[dtype])
    return np.exp2(np.floor(np.log2(a)) - mant)


def assert_close_rounded(got, ref, dtype, what=""):
    """Causal rows near a prompt's start average few values, so |out| reaches
    ~4 where half an ulp of bf16 alone is 8e-3 to 1.6e-2.  Bound: each output
    within 1e-2 plus half an ulp of its exact value; mean |error| <= 1e-3."""
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    err = np.abs(got - ref)
    excess = err - (MAX_ABS + half_ulp(ref, dtype))
    i = np.unravel_index(np.argmax(excess), err.shape)
    assert excess.max() <= 0, (f"{what}: |err| {err[i]:.3e} at {i} (ref {ref[i]:.4f}, got "
                               f"{got[i]:.4f}) beyond 1e-2 + half ulp")
    assert err.mean() <= MEAN_ABS, f"{what}: mean {err.mean():.3e}"
    return float(err.max()), float(err.mean())
