"""Block-move oracle checked by brute force on tiny pools: every element of every block is
where the copy-on-write copy or the offload gather / restore scatter says it must be."""
import numpy as np
import pytest

from oracle import blocks as ob


def _pool(P=6, bs=4, H=2, D=3, seed=0):
    return np.random.default_rng(seed).integers(0, 1 << 16, (P, bs, H, D), dtype=np.uint16)


def test_copy_blocks_elementwise():
    pool = _pool()
    out = ob.copy_blocks(pool, [1, 4], [3, 0])
    P, bs, H, D = pool.shape
    for b in range(P):
        for t in range(bs):
            for h in range(H):
                for d in range(D):
                    want = pool[{3: 1, 0: 4}.get(b, b), t, h, d]
                    assert out[b, t, h, d] == want
    assert (pool == _pool()).all()                     # input untouched


def test_copy_same_block_is_a_noop_and_overlap_is_rejected():
    pool = _pool()
    assert (ob.copy_blocks(pool, [2], [2]) == pool).all()
    with pytest.raises(ValueError):
        ob.copy_blocks(pool, [1, 2], [2, 3])           # block 2 both read and written


def test_gather_then_scatter_elsewhere_moves_blocks():
    pool = _pool()
    host = ob.gather_blocks(pool, [5, 0, 2])
    assert host.shape == (3,) + pool.shape[1:]
    for i, b in enumerate([5, 0, 2]):
        assert (host[i] == pool[b]).all()
    back = ob.scatter_blocks(pool, [1, 3, 4], host)
    for i, b in enumerate([1, 3, 4]):
        assert (back[b] == pool[[5, 0, 2][i]]).all()
    for b in (0, 2, 5):
        assert (back[b] == pool[b]).all()
    assert ob.gather_blocks(pool, []).shape == (0,) + pool.shape[1:]
