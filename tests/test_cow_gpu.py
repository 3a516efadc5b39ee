"""Copy-on-write on the GPU: pa_copy_blocks byte-identical to the oracle's
block copy, and a fork inside a block carried end to end -- the product
allocator's slots and copy pairs, pa_copy_blocks, pa_cache_write and
pa_decode -- against the oracle replaying the same steps with its own
allocator model."""
import numpy as np
import pytest
import torch

import gpu_util as U
import oracle
from oracle.allocator import AllocatorModel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return U.require_gpu()


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_copy_blocks_bit_exact(pa):
    b = U.batch("llama8b")
    Lr = b.layers[0]
    rng = np.random.default_rng(4)
    ids = rng.permutation(b.num_blocks)
    src = ids[:40].astype(np.int32)
    dst = ids[40:80].astype(np.int32)
    src[3], dst[7] = b.num_blocks + 2, -1          # outside the pool: skipped
    kd, vd = U.to_dev(Lr.k_cache, "bf16").clone(), U.to_dev(Lr.v_cache, "bf16").clone()
    pa.pa_copy_blocks(kd, vd, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    torch.cuda.synchronize()
    ok, ov, skipped = oracle.copy_blocks(_u16(Lr.k_cache), _u16(Lr.v_cache), src, dst)
    assert skipped == 2
    assert np.array_equal(_u16(kd), ok) and np.array_equal(_u16(vd), ov)


def test_fork_inside_a_block_end_to_end(pa):
    """Parent of 40 tokens (3 blocks, the last holding 8); a child forked at
    40 shares all three.  Both append one token: the child's write into the
    shared partial block copies it first; the parent's does not.  A second
    child forked at 32 shares only full blocks."""
    H, Hq, D, bs = 8, 32, 128, 16
    nb = 24
    scale = 1.0 / np.sqrt(D)
    order = np.random.default_rng(11).permutation(nb).astype(np.int32)
    A = pa.Allocator(nb, order)
    M = AllocatorModel(nb, bs, order)
    g = torch.Generator().manual_seed(12)
    rand = lambda *s: torch.randn(s, generator=g).to(torch.bfloat16)

    kc = torch.full((nb, H, bs, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    okc, ovc = _u16(kc), _u16(vc)

    def write(slots, k, v):
        nonlocal okc, ovc
        pa.pa_cache_write(k.cuda(), v.cuda(), torch.tensor(slots, dtype=torch.int64).cuda(), kc, vc)
        okc, ovc, bad = oracle.cache_write(_u16(k), _u16(v), np.array(slots, np.int64), okc, ovc)
        assert bad == 0

    p, mp = A.seq_create(), M.seq_create()
    slots, cow = A.append_slots([p], 40)
    mslots, mcow = M.append_slots([mp], 40)
    assert slots == mslots and cow == mcow == []
    write(slots, rand(40, H, D), rand(40, H, D))
    c1, mc1 = A.seq_fork(p, 40), M.seq_fork(mp, 40)
    c2, mc2 = A.seq_fork(p, 32), M.seq_fork(mp, 32)
    slots, cow = A.append_slots([c1, p, c2], 1)
    mslots, mcow = M.append_slots([mc1, mp, mc2], 1)
    assert slots == mslots and cow == mcow and len(cow) == 1
    src = torch.tensor([cow[0][0]], dtype=torch.int32).cuda()
    dst = torch.tensor([cow[0][1]], dtype=torch.int32).cuda()
    pa.pa_copy_blocks(kc, vc, src, dst)
    okc, ovc, _ = oracle.copy_blocks(okc, ovc, [cow[0][0]], [cow[0][1]])
    write(slots, rand(3, H, D), rand(3, H, D))
    torch.cuda.synchronize()
    assert np.array_equal(_u16(kc), okc) and np.array_equal(_u16(vc), ovc)

    seqs = [p, c1, c2]
    rows, lens = A.block_table(seqs, 4)
    assert lens == [41, 41, 33]
    mrows, mlens = M.block_table(seqs, 4)
    assert rows == mrows and lens == mlens
    st = A.stats()
    assert st["shared"] == 2 and st["refs"] == 3 + 3 + 3   # blocks 0, 1 shared by all three
    q = rand(3, Hq, D)
    tab = np.array([[x if x >= 0 else 0 for x in r] for r in rows], np.int32)
    out = pa.pa_decode(q.cuda(), kc, vc, torch.from_numpy(tab).cuda(),
                       torch.tensor(lens, dtype=torch.int32).cuda(), scale)
    torch.cuda.synchronize()
    ref = oracle.decode(_u16(q), okc, ovc, tab, np.array(lens, np.int32), scale, "bf16")
    U.assert_close(out.double().cpu().numpy(), ref, "fork inside a block")
    # the child and the parent share 40 tokens but not the 41st: outputs differ
    assert not np.allclose(ref[0], ref[1])
