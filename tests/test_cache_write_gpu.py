"""pa_cache_write on the GPU: byte-identical to the oracle's scatter."""
import numpy as np
import pytest
import torch

import gpu_util as U
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def gpu_write(pa, b, k, v, slots, kc, vc):
    w = b.workload
    kd, vd = U.to_dev(kc, w.dtype).clone(), U.to_dev(vc, w.dtype).clone()
    pa.pa_cache_write(U.to_dev(k, w.dtype), U.to_dev(v, w.dtype), torch.from_numpy(slots).cuda(),
                      kd, vd)
    torch.cuda.synchronize()
    return kd.view(torch.int16).cpu().numpy().view(np.uint16), \
        vd.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["tiny", "llama8b", "llama70b", "long", "fullstep"])
def test_new_tokens_bit_exact(pa, name):
    b = U.batch(name, num_layers=1) if name == "fullstep" else U.batch(name)
    Lr = b.layers[0]
    gk, gv = gpu_write(pa, b, Lr.new_k, Lr.new_v, b.slot_mapping, Lr.k_cache, Lr.v_cache)
    ok, ov, bad = oracle.cache_write(Lr.new_k.numpy().view(np.uint16),
                                     Lr.new_v.numpy().view(np.uint16), b.slot_mapping,
                                     Lr.k_cache.numpy().view(np.uint16),
                                     Lr.v_cache.numpy().view(np.uint16))
    assert bad == 0
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_padding_out_of_range_and_many_tokens(pa):
    b = U.batch("llama8b")
    w = b.workload
    rng = np.random.default_rng(1)
    T = 3000
    slots = rng.choice(b.num_blocks * 16, size=T, replace=False).astype(np.int64)
    slots[::7] = -1
    slots[5] = b.num_blocks * 16 + 3        # past the pool: not written
    gen = torch.Generator().manual_seed(2)
    k = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen).to(torch.bfloat16).view(torch.int16)
    v = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen).to(torch.bfloat16).view(torch.int16)
    Lr = b.layers[0]
    gk, gv = gpu_write(pa, b, k, v, slots, Lr.k_cache, Lr.v_cache)
    ok, ov, bad = oracle.cache_write(k.numpy().view(np.uint16), v.numpy().view(np.uint16), slots,
                                     Lr.k_cache.numpy().view(np.uint16),
                                     Lr.v_cache.numpy().view(np.uint16))
    assert bad == 1
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_fp16_head_dim_64(pa):
    b = U.batch("tiny")
    w = b.workload
    slots = np.array([3, -1, 24 * 16 - 1, 100], np.int64)
    gen = torch.Generator().manual_seed(3)
    k = torch.randn((4, 2, 64), generator=gen).to(torch.float16).view(torch.int16)
    v = torch.randn((4, 2, 64), generator=gen).to(torch.float16).view(torch.int16)
    Lr = b.layers[0]
    gk, gv = gpu_write(pa, b, k, v, slots, Lr.k_cache, Lr.v_cache)
    ok, ov, _ = oracle.cache_write(k.numpy().view(np.uint16), v.numpy().view(np.uint16), slots,
                                   Lr.k_cache.numpy().view(np.uint16),
                                   Lr.v_cache.numpy().view(np.uint16))
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
