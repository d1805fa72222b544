"""Seeded random ragged batches through the CUDA path, element by element against the oracle:
decode tokens, chunks of many lengths (ragged last tiles), empty sequences, GQA groups 1-8,
head dims 64 and 128, block sizes 4-64, shuffled pages, sliding windows on some batches, and the
one-call append + attention entry on others."""
import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from gpu_util import DeviceBatch, assert_close, bits_of, oracle_append
from oracle import paged_attention as opa

pytestmark = pytest.mark.gpu


def _random_batch(trial):
    rng = np.random.default_rng(9000 + trial)
    S = int(rng.integers(1, 24))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([4, 16, 32, 64]))
    q_lens, kv_lens = [], []
    for _ in range(S):
        kind = rng.random()
        q = 0 if kind < 0.1 else 1 if kind < 0.6 else int(rng.integers(2, 300))
        ctx = int(rng.integers(0, 1500))
        q_lens.append(q)
        kv_lens.append(max(q + ctx, 1) if q == 0 else q + ctx)
    b = workloads.build_batch(q_lens, kv_lens, G * Hkv, Hkv, D, bs, seed=9100 + trial,
                              shuffle_pages=True, name=f"random {trial}")
    window = int(rng.choice([0, 0, 0, 64, 300]))
    return b, window


@pytest.mark.parametrize("trial", range(10))
def test_random_ragged_batch_matches_oracle(cuda_lib, trial):
    b, window = _random_batch(trial)
    db = DeviceBatch(b)
    fused = trial % 2 == 1
    if fused:
        out = cb.append_attention(db.q, db.k_new, db.v_new, db.k_pages, db.v_pages,
                                  db.block_table, db.cu, db.kv_lens, b.block_size, b.scale,
                                  window=window)
    else:
        db.append()
        out = cb.ragged_paged_attention(db.q, db.k_pages, db.v_pages, db.block_table, db.cu,
                                        db.kv_lens, b.block_size, b.scale, window=window)
    assert cb.get_device_error() == cb.CB_OK
    kp, vp = oracle_append(b)
    assert np.array_equal(bits_of(db.k_pages), kp) and np.array_equal(bits_of(db.v_pages), vp)
    ref, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                        b.block_size, b.scale, window=window)
    assert_close(out.float().cpu().numpy(), ref, f"{b.name} (window {window}, fused {fused})")


@pytest.mark.parametrize("G", [4, 3])
def test_many_one_tile_chunk_items(cuda_lib, G):
    """Hundreds of chunk work items of one K/V tile each (short chunks at short prior contexts,
    with decodes between them): every chunk CTA runs many items back to back, so the next item
    is claimed at an item's first stage and the two decoded-item slots turn over quickly.  With
    an odd group size an item pairs two query tiles of one head; some chunks span two tiles."""
    rng = np.random.default_rng(9400 + G)
    q_lens, kv_lens = [], []
    for i in range(360):
        if i % 5 == 4:
            q, ctx = 1, int(rng.integers(1, 200))
        else:
            q = int(rng.integers(2, 60)) if i % 7 else int(rng.integers(120, 250))
            ctx = int(rng.integers(0, 128 - min(q, 127)))
        q_lens.append(q)
        kv_lens.append(q + ctx)
    Hkv = 2
    b = workloads.build_batch(q_lens, kv_lens, G * Hkv, Hkv, 128, 16, seed=9450 + G,
                              shuffle_pages=True, name=f"one-tile items G {G}")
    db = DeviceBatch(b)
    out = cb.append_attention(db.q, db.k_new, db.v_new, db.k_pages, db.v_pages, db.block_table,
                              db.cu, db.kv_lens, b.block_size, b.scale)
    assert cb.get_device_error() == cb.CB_OK
    kp, vp = oracle_append(b)
    ref, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                        b.block_size, b.scale)
    assert_close(out.float().cpu().numpy(), ref, b.name)


def _wide_batch(trial):
    """Wider random mix than _random_batch: GQA groups up to 16 (two warps per KV head in the
    decode pass), odd groups, block sizes 4-128, explicit decode CTA counts, and every fourth
    batch hundreds of short sequences (many decode parts and one-tile chunk items)."""
    rng = np.random.default_rng(77000 + trial)
    many = trial % 4 == 3
    S = int(rng.integers(100, 400)) if many else int(rng.integers(1, 60))
    G = int(rng.choice([1, 2, 3, 4, 8, 12, 16]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    if G > 8:
        Hkv = min(Hkv, 4)
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([4, 8, 16, 32, 64, 128]))
    q_lens, kv_lens = [], []
    for _ in range(S):
        u = rng.random()
        if many:
            q = 1 if u < 0.3 else int(rng.integers(2, 80))
            ctx = int(rng.integers(0, 200))
        else:
            q = 0 if u < 0.05 else 1 if u < 0.55 else int(rng.integers(2, 400))
            ctx = int(rng.integers(0, 3000))
        q_lens.append(q)
        kv_lens.append(max(q + ctx, 1) if q == 0 else q + ctx)
    window = int(rng.choice([0, 0, 0, 0, 32, 200, 1000]))
    decode_ctas = int(rng.choice([0, 0, 0, 1, 5, 40, 200]))
    fused = bool(rng.integers(0, 2))
    b = workloads.build_batch(q_lens, kv_lens, G * Hkv, Hkv, D, bs, seed=78000 + trial,
                              shuffle_pages=True, name=f"wide random {trial}")
    return b, window, decode_ctas, fused


@pytest.mark.parametrize("trial", range(24))
def test_wide_random_batch_matches_oracle(cuda_lib, trial):
    b, window, decode_ctas, fused = _wide_batch(trial)
    db = DeviceBatch(b)
    kw = dict(window=window, decode_ctas=decode_ctas)
    if fused:
        out = cb.append_attention(db.q, db.k_new, db.v_new, db.k_pages, db.v_pages,
                                  db.block_table, db.cu, db.kv_lens, b.block_size, b.scale, **kw)
    else:
        db.append()
        out = cb.ragged_paged_attention(db.q, db.k_pages, db.v_pages, db.block_table, db.cu,
                                        db.kv_lens, b.block_size, b.scale, **kw)
    assert cb.get_device_error() == cb.CB_OK
    kp, vp = oracle_append(b)
    assert np.array_equal(bits_of(db.k_pages), kp) and np.array_equal(bits_of(db.v_pages), vp)
    ref, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                        b.block_size, b.scale, window=window)
    assert_close(out.float().cpu().numpy(), ref,
                 f"{b.name} (window {window}, decode_ctas {decode_ctas}, fused {fused})")
