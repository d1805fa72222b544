"""The seeded input recipe (workloads.py) produces the named batches the design describes: the
lengths, head shapes, block sizes and sharing of each, and the poisoning of every slot outside a
sequence's visible keys."""
import numpy as np
import pytest

import workloads


def _lens(n):
    return workloads.config_lengths(n, 1000 + n)


def test_tiny_ragged_batch():
    q, kv, kw = _lens(1)
    assert q == [32, 1, 1, 1] and kv == [32, 18, 65, 101]       # prior context 0 / 17 / 64 / 100
    assert (kw["num_q_heads"], kw["num_kv_heads"], kw["head_dim"], kw["block_size"],
            kw["num_pages"], kw["scale"]) == (4, 2, 64, 16, 24, 1.0 / 8.0)


def test_decode_only_batch():
    q, kv, kw = _lens(2)
    assert q == [1] * 64 and len(kv) == 64 and kv.min() >= 512 and kv.max() <= 4096
    assert (kw["num_q_heads"], kw["num_kv_heads"], kw["head_dim"], kw["block_size"],
            kw["num_pages"]) == (32, 8, 128, 32, 16384)


def test_mixed_batch_fills_the_token_budget():
    q, kv, kw = _lens(3)
    assert q[:120] == [1] * 120 and q[120] == 1928 and sum(q) == 2048
    ctx = np.asarray(kv) - np.asarray(q)
    assert ctx[:120].min() >= 256 and ctx[:120].max() <= 8192 and ctx[120] == 3000
    assert (kw["num_q_heads"], kw["num_kv_heads"], kw["head_dim"], kw["block_size"]) == (32, 8, 128, 32)


def test_chunk_heavy_batch():
    q, kv, kw = _lens(4)
    assert q == [1] * 16 + [512] * 8 and sum(q) == 4112
    ctx = np.asarray(kv) - np.asarray(q)
    assert ctx.min() >= 0 and ctx.max() <= 8192
    assert kw["block_size"] == 64 and kw["k_scale"] == 4.0


def test_long_tail_batch_with_a_shared_prefix():
    q, kv, kw = _lens(5)
    kv = np.asarray(kv)
    assert q == [1] * 256 and kv.max() <= 32768 and kv.min() >= 1
    assert 1500 <= np.median(kv) <= 2800                        # lognormal around 2048
    members, n_tok = kw["shared_prefix"]
    assert members == list(range(64)) and n_tok == 1024 and n_tok % kw["block_size"] == 0
    assert kv[:64].min() >= 1025                                # the new token lands past the prefix
    assert (kw["num_q_heads"], kw["num_kv_heads"], kw["block_size"]) == (64, 8, 64)


def test_shared_prefix_members_point_at_the_same_pages():
    b = workloads.build_batch([1, 1, 1], [40, 37, 50], 4, 2, 8, 4, seed=3,
                              shared_prefix=([0, 1], 32))
    assert np.array_equal(b.block_table[0, :8], b.block_table[1, :8])
    assert not np.intersect1d(b.block_table[2][b.block_table[2] >= 0], b.block_table[0, :8]).size
    used = b.block_table[b.block_table >= 0]
    assert len(np.unique(used)) == len(used) - 8                  # only the prefix is shared


@pytest.mark.parametrize("seed", [1, 2])
def test_slots_outside_the_prior_context_are_poisoned(seed):
    b = workloads.build_batch([3, 1, 0], [10, 7, 5], 4, 2, 8, 4, seed=seed)
    k = b.k_pages.reshape(-1, 2, 8)
    nan_bits = (k & 0x7F80) == 0x7F80
    q_lens = np.diff(b.cu_seqlens_q)
    visible = np.zeros(k.shape[0], dtype=bool)
    for s in range(b.num_seqs):
        ctx = int(b.kv_lens[s]) - int(q_lens[s])
        for p in range(ctx):
            visible[b.block_table[s][p // 4] * 4 + p % 4] = True
    assert not nan_bits[visible].any()                            # prior context holds values
    assert nan_bits[~visible].all()                               # everything else is NaN
