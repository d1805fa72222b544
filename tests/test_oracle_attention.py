"""Pins of the attention / append oracle against things other than itself.

No page prints an attention output, so the oracle is pinned by an independent
library routine (torch's scaled_dot_product_attention in float64), closed
forms, explicit Python-float loops on tiny inputs, and the invariants the
method must satisfy (ragged == alone, page permutation, prefix sharing,
convexity, softmax shift invariance).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import workloads
from oracle import paged_attention as opa
from oracle.paged_attention import OracleError


def _f64(bits):
    return opa.bf16_bits_to_f64(bits)


def _appended(b):
    return opa.kv_append(b.k_new, b.v_new, b.k_pages, b.v_pages, b.block_table,
                         b.cu_seqlens_q, b.kv_lens, b.block_size)


def _attend(b, kp, vp, table=None):
    return opa.ragged_paged_attention(b.q, kp, vp, b.block_table if table is None else table,
                                      b.cu_seqlens_q, b.kv_lens, b.block_size, b.scale)


# ----------------------------------------------------------------------------- conversions

def test_bf16_conversion_exact_values():
    bits = np.array([0x3F80, 0xBF80, 0x4000, 0x0000, 0x3E80, 0x7F80], dtype=np.uint16)
    assert list(_f64(bits)) == [1.0, -1.0, 2.0, 0.0, 0.25, math.inf]
    # round trip with the generator's rounding on values bf16 holds exactly
    x = np.array([1.5, -3.0, 0.0078125, 96.0], dtype=np.float32)
    assert np.array_equal(_f64(workloads.f32_to_bf16_bits(x)), x.astype(np.float64))


# ----------------------------------------------------------------------------- append

def test_append_worked_example_slot():
    # Block size 4, A's table [7, 2, 5]: token 9 is in block 5 at offset 1.  A has 9 prior
    # tokens and appends one token (position 9); every other slot stays as it was.
    P, bs, Hkv, D = 8, 4, 1, 2
    kp = np.zeros((P, bs, Hkv, D), dtype=np.uint16)
    vp = np.zeros_like(kp)
    k_new = np.array([[[0x1111, 0x2222]]], dtype=np.uint16)
    v_new = np.array([[[0x3333, 0x4444]]], dtype=np.uint16)
    table = np.array([[7, 2, 5]], dtype=np.int32)
    k2, v2 = opa.kv_append(k_new, v_new, kp, vp, table, [0, 1], [10], bs)
    flat_k = k2.reshape(P * bs, Hkv, D)
    changed = np.nonzero(np.any(flat_k != 0, axis=(1, 2)))[0]
    assert list(changed) == [21]
    assert list(k2[5, 1, 0]) == [0x1111, 0x2222] and list(v2[5, 1, 0]) == [0x3333, 0x4444]


@pytest.mark.parametrize("cfg", [1, "mixed"])
def test_append_inverse_map(cfg):
    """Every written slot maps back to exactly the (sequence, position) that wrote it."""
    if cfg == "mixed":
        b = workloads.build_batch([1, 40, 1, 0, 17], [9, 40, 33, 5, 50], 4, 2, 8, 4, seed=12)
    else:
        b = workloads.make_config(cfg)
    k2, _ = _appended(b)
    P, bs = b.num_pages, b.block_size
    flat_old = b.k_pages.reshape(P * bs, -1)
    flat_new = k2.reshape(P * bs, -1)
    changed = set(np.nonzero(np.any(flat_old != flat_new, axis=1))[0].tolist())
    expect = {}
    for s in range(b.num_seqs):
        ql = int(b.q_lens[s])
        ctx = int(b.kv_lens[s]) - ql
        row = list(b.block_table[s])
        for i in range(ql):
            pos = ctx + i
            # inverse: find the logical block whose physical id holds this slot
            expect_slot = row[pos // bs] * bs + pos % bs
            expect[expect_slot] = int(b.cu_seqlens_q[s]) + i
    assert changed == set(expect)
    for slot, t in expect.items():
        blk, off = divmod(slot, bs)
        s = int(np.searchsorted(b.cu_seqlens_q, t, side="right") - 1)
        j = list(b.block_table[s]).index(blk)
        assert j * bs + off == int(b.kv_lens[s]) - int(b.q_lens[s]) + (t - int(b.cu_seqlens_q[s]))
        assert np.array_equal(flat_new[slot], b.k_new[t].reshape(-1))


def test_append_rejects_undefined_metadata():
    b = workloads.build_batch([2, 1], [5, 3], 2, 1, 8, 4, seed=3)
    args = (b.k_new, b.v_new, b.k_pages, b.v_pages)
    bad_table = b.block_table.copy()
    bad_table[0, 1] = b.num_pages  # outside the pool
    with pytest.raises(OracleError):
        opa.kv_append(*args, bad_table, b.cu_seqlens_q, b.kv_lens, 4)
    with pytest.raises(OracleError):
        opa.kv_append(*args, b.block_table, b.cu_seqlens_q, [1, 3], 4)  # kv_len < q_len
    with pytest.raises(OracleError):
        opa.kv_append(*args, b.block_table, [0, 2, 1], b.kv_lens, 4)   # decreasing cu
    dup = b.block_table.copy()
    dup[1, 0] = dup[0, 1]  # seq 1's block aliases seq 0's second block
    with pytest.raises(OracleError):
        opa.kv_append(*args, dup, b.cu_seqlens_q, b.kv_lens, 4)
    with pytest.raises(OracleError):
        opa.kv_append(*args, b.block_table, b.cu_seqlens_q, b.kv_lens, 3)  # block_size < 4


# ----------------------------------------------------------------------------- attention pins

def test_softmax_shift_invariance_and_lse():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 17)) * 3
    p0, l0 = opa.stable_softmax(x, axis=1)
    for c in (1e4, -1e4, 37.5):
        p1, l1 = opa.stable_softmax(x + c, axis=1)
        assert np.allclose(p1, p0, rtol=0, atol=1e-9)
        assert np.allclose(l1 - c, l0, rtol=0, atol=1e-8)
    assert np.allclose(l0, scipy.special.logsumexp(x, axis=1), rtol=0, atol=1e-12)
    assert np.allclose(p0, scipy.special.softmax(x, axis=1), rtol=0, atol=1e-15)


def _single_sequence(n_q, kv, Hq, Hkv, D, bs, seed, shuffle=False):
    b = workloads.build_batch([n_q], [kv], Hq, Hkv, D, bs, seed=seed, shuffle_pages=shuffle)
    kp, vp = _appended(b)
    return b, kp, vp


@pytest.mark.parametrize("bs", [4, 16])
def test_dense_causal_matches_sdpa(bs):
    """One sequence with ctx 0: textbook causal attention (library routine, float64)."""
    n, H, D = 23, 3, 16
    b, kp, vp = _single_sequence(n, n, H, H, D, bs, seed=11, shuffle=True)
    out, lse = _attend(b, kp, vp)
    K = opa.gather_kv(kp, b.block_table[0], n, bs)
    V = opa.gather_kv(vp, b.block_table[0], n, bs)
    q = torch.from_numpy(_f64(b.q)).permute(1, 0, 2)      # [H, n, D]
    k = torch.from_numpy(K).permute(1, 0, 2)
    v = torch.from_numpy(V).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=b.scale)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    # lse against scipy's logsumexp over the visible scores
    s = np.einsum("hid,hjd->hij", q.numpy(), k.numpy()) * b.scale
    mask = np.tril(np.ones((n, n), dtype=bool))
    lref = scipy.special.logsumexp(np.where(mask, s, -np.inf), axis=2).T
    assert np.allclose(lse, lref, rtol=0, atol=1e-12)


def test_chunk_equals_tail_of_full_prefill():
    """A chunk at prior context ctx returns the last rows of a full causal prefill of ctx+n tokens."""
    ctx, n, H, D, bs = 37, 13, 2, 8, 16
    b, kp, vp = _single_sequence(n, ctx + n, H, H, D, bs, seed=5, shuffle=True)
    out, _ = _attend(b, kp, vp)
    K = torch.from_numpy(opa.gather_kv(kp, b.block_table[0], ctx + n, bs)).permute(1, 0, 2)
    V = torch.from_numpy(opa.gather_kv(vp, b.block_table[0], ctx + n, bs)).permute(1, 0, 2)
    # full prefill queries: arbitrary rows for the first ctx positions, the chunk's after
    rng = np.random.default_rng(1)
    full_q = np.concatenate([rng.standard_normal((ctx, H, D)), _f64(b.q)], axis=0)
    qf = torch.from_numpy(full_q).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qf, K, V, is_causal=True, scale=b.scale)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy()[ctx:], rtol=0, atol=1e-12)


def test_closed_forms():
    # kv_len == 1: the only visible value row comes back unchanged.
    b, kp, vp = _single_sequence(1, 1, 4, 2, 8, 4, seed=2)
    out, lse = _attend(b, kp, vp)
    v0 = opa.gather_kv(vp, b.block_table[0], 1, 4)[0]
    assert np.array_equal(out[0], np.repeat(v0, 2, axis=0))
    # q == 0: uniform weights, out = mean of the visible V rows, lse = log(#visible).
    b, kp, vp = _single_sequence(5, 12, 2, 2, 8, 4, seed=3)
    b.q[:] = 0
    out, lse = _attend(b, kp, vp)
    V = opa.gather_kv(vp, b.block_table[0], 12, 4)
    for i in range(5):
        vis = 12 - 5 + i + 1
        assert np.allclose(out[i], V[:vis].mean(axis=0), rtol=0, atol=1e-14)
        assert np.allclose(lse[i], math.log(vis), rtol=0, atol=1e-14)
    # identical keys: every score is equal, so the result is again the mean of V.
    b, kp, vp = _single_sequence(3, 9, 2, 1, 8, 4, seed=4)
    kp[...] = kp[b.block_table[0, 0], 0, 0][None, None, None, :]
    out, _ = _attend(b, kp, vp)
    V = opa.gather_kv(vp, b.block_table[0], 9, 4)
    for i in range(3):
        assert np.allclose(out[i], V[: 9 - 3 + i + 1].mean(axis=0)[0][None, :], atol=1e-14)


def _brute_force(q, kp, vp, table, cu, kv_lens, bs, scale):
    """Explicit loops over Python floats: the definition with nothing vectorised."""
    T, Hq, D = len(q), len(q[0]), len(q[0][0])
    Hkv = len(kp[0][0])
    G = Hq // Hkv
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(T)]
    for s in range(len(kv_lens)):
        n = cu[s + 1] - cu[s]
        ctx = kv_lens[s] - n
        for i in range(n):
            t = cu[s] + i
            for h in range(Hq):
                g = h // G
                scores = []
                for j in range(ctx + i + 1):
                    blk = table[s][j // bs]
                    kj = kp[blk][j % bs][g]
                    scores.append(scale * sum(float(q[t][h][d]) * float(kj[d]) for d in range(D)))
                m = max(scores)
                w = [math.exp(x - m) for x in scores]
                z = sum(w)
                for d in range(D):
                    acc = 0.0
                    for j, wj in enumerate(w):
                        blk = table[s][j // bs]
                        acc += wj * float(vp[blk][j % bs][g][d])
                    out[t][h][d] = acc / z
    return np.array(out)


def test_brute_force_tiny():
    b = workloads.build_batch([3, 1, 2], [5, 8, 2], 4, 2, 4, 4, seed=9)
    kp, vp = _appended(b)
    out, _ = _attend(b, kp, vp)
    ref = _brute_force(_f64(b.q).tolist(), _f64(kp).tolist(), _f64(vp).tolist(),
                       b.block_table.tolist(), b.cu_seqlens_q.tolist(), b.kv_lens.tolist(),
                       b.block_size, b.scale)
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- invariants

def test_ragged_equals_each_sequence_alone():
    b = workloads.make_config(1)
    kp, vp = _appended(b)
    out, lse = _attend(b, kp, vp)
    for s in range(b.num_seqs):
        a, e = int(b.cu_seqlens_q[s]), int(b.cu_seqlens_q[s + 1])
        o1, l1 = opa.ragged_paged_attention(b.q[a:e], kp, vp, b.block_table[s:s + 1],
                                            [0, e - a], b.kv_lens[s:s + 1], b.block_size, b.scale)
        assert np.array_equal(o1, out[a:e]) and np.array_equal(l1, lse[a:e])


def test_page_permutation_invariance():
    b = workloads.make_config(1)
    kp, vp = _appended(b)
    out, lse = _attend(b, kp, vp)
    perm = np.random.default_rng(3).permutation(b.num_pages)   # new id of old page i is perm[i]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    table2 = np.where(b.block_table >= 0, perm[np.maximum(b.block_table, 0)], -1)
    out2, lse2 = _attend(b, kp2, vp2, table2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_shared_prefix_equals_duplicated_copy():
    q_lens = [1, 1, 2]
    kv = [70, 90, 66]
    b = workloads.build_batch(q_lens, kv, 4, 2, 8, 16, seed=21,
                              shared_prefix=([0, 1, 2], 64))
    assert b.block_table[0, 0] == b.block_table[1, 0] == b.block_table[2, 0]
    kp, vp = _appended(b)
    out, lse = _attend(b, kp, vp)
    # Duplicate the shared blocks into fresh pages for sequences 1 and 2.
    n_sh = 64 // 16
    extra = 2 * n_sh
    P = b.num_pages
    kp2 = np.concatenate([kp, np.zeros((extra,) + kp.shape[1:], np.uint16)])
    vp2 = np.concatenate([vp, np.zeros((extra,) + vp.shape[1:], np.uint16)])
    table2 = b.block_table.copy()
    for r, s in enumerate((1, 2)):
        for j in range(n_sh):
            new = P + r * n_sh + j
            kp2[new] = kp[table2[s, j]]
            vp2[new] = vp[table2[s, j]]
            table2[s, j] = new
    out2, lse2 = _attend(b, kp2, vp2, table2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_output_in_convex_hull_of_visible_values():
    b = workloads.make_config(1)
    kp, vp = _appended(b)
    out, _ = _attend(b, kp, vp)
    G = b.num_q_heads // b.num_kv_heads
    for s in range(b.num_seqs):
        V = opa.gather_kv(vp, b.block_table[s], int(b.kv_lens[s]), b.block_size)
        n = int(b.q_lens[s])
        ctx = int(b.kv_lens[s]) - n
        for i in range(n):
            t = int(b.cu_seqlens_q[s]) + i
            for h in range(b.num_q_heads):
                vis = V[: ctx + i + 1, h // G]
                assert np.all(out[t, h] >= vis.min(axis=0) - 1e-12)
                assert np.all(out[t, h] <= vis.max(axis=0) + 1e-12)


def test_poison_is_never_read():
    """The generator poisons every slot outside the visible keys; no NaN may reach the output."""
    for cfg in (1,):
        b = workloads.make_config(cfg)
        kp, vp = _appended(b)
        out, lse = _attend(b, kp, vp)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
    # ... and skipping the append leaves the new tokens' slots poisoned.
    b = workloads.make_config(1)
    out, _ = _attend(b, b.k_pages, b.v_pages)
    assert np.isnan(out).any()


def test_attention_rows_matches_full():
    b = workloads.make_config(1)
    kp, vp = _appended(b)
    out, lse = _attend(b, kp, vp)
    rows = [(0, 0), (5, 3), (31, 1), (32, 2), (34, 3)]
    o, l = opa.attention_rows(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                              b.block_size, b.scale, rows)
    for r, (t, h) in enumerate(rows):
        assert np.allclose(o[r], out[t, h], rtol=0, atol=1e-12)
        assert np.allclose(l[r], lse[t, h], rtol=0, atol=1e-12)


def test_zero_length_sequences_are_noops():
    b = workloads.build_batch([0, 3, 0], [4, 6, 0], 2, 1, 8, 4, seed=8)
    kp, vp = _appended(b)
    out, _ = _attend(b, kp, vp)
    assert out.shape == (3, 2, 8) and np.isfinite(out).all()


def test_gather_matches_scalar_slot_rule():
    b = workloads.make_config(1)
    for s in range(b.num_seqs):
        K = opa.gather_kv(b.k_pages, b.block_table[s], int(b.kv_lens[s]), b.block_size)
        flat = b.k_pages.reshape(b.num_pages * b.block_size, *b.k_pages.shape[2:])
        for j in range(int(b.kv_lens[s])):
            slot = opa.slot_of(b.block_table[s], j, b.block_size, b.num_pages)
            assert np.array_equal(K[j], _f64(flat[slot]), equal_nan=True)
    with pytest.raises(OracleError):
        opa.gather_kv(b.k_pages, b.block_table[0], 10 ** 4, b.block_size)


# ----------------------------------------------------------------------------- sliding window

@pytest.mark.parametrize("window", [1, 3, 16, 40])
def test_sliding_window_matches_sdpa_with_a_band_mask(window):
    """Sliding window W: query at position p sees keys (p - W, p].  Against the library
    attention routine with the equivalent boolean band mask (float64)."""
    ctx, n, H, D, bs = 30, 17, 2, 8, 4
    b, kp, vp = _single_sequence(n, ctx + n, H, H, D, bs, seed=21, shuffle=True)
    cu, kv = b.cu_seqlens_q, b.kv_lens
    out, lse = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, cu, kv, bs, b.scale,
                                          window=window)
    K = torch.from_numpy(opa.gather_kv(kp, b.block_table[0], ctx + n, bs)).permute(1, 0, 2)
    V = torch.from_numpy(opa.gather_kv(vp, b.block_table[0], ctx + n, bs)).permute(1, 0, 2)
    q = torch.from_numpy(_f64(b.q)).permute(1, 0, 2)
    pos = torch.arange(ctx, ctx + n)[:, None]
    keys = torch.arange(ctx + n)[None, :]
    band = (keys <= pos) & (keys > pos - window)
    ref = torch.nn.functional.scaled_dot_product_attention(q, K, V, attn_mask=band, scale=b.scale)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    rows = [(t, h) for t in range(n) for h in range(H)]
    ro, rl = opa.attention_rows(b.q, kp, vp, b.block_table, cu, kv, bs, b.scale, rows, window=window)
    assert np.allclose(ro, out.reshape(-1, D), rtol=0, atol=1e-12)
    assert np.allclose(rl, lse.reshape(-1), rtol=0, atol=1e-12)


def test_sliding_window_closed_forms():
    ctx, n, H, D, bs = 9, 5, 2, 4, 4
    b, kp, vp = _single_sequence(n, ctx + n, H, H, D, bs, seed=22, shuffle=False)
    K = opa.gather_kv(kp, b.block_table[0], ctx + n, bs)
    V = opa.gather_kv(vp, b.block_table[0], ctx + n, bs)
    # W = 1: every query sees only its own key, so out = its own value row
    out, lse = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                          bs, b.scale, window=1)
    for i in range(n):
        assert np.allclose(out[i], V[ctx + i], rtol=0, atol=1e-12)
        assert np.allclose(lse[i], b.scale * np.sum(_f64(b.q)[i] * K[ctx + i], axis=-1), atol=1e-12)
    # a window at least as long as the sequence is the full causal pass
    full, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                         bs, b.scale)
    wide, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                         bs, b.scale, window=ctx + n)
    assert np.array_equal(full, wide)


# ----------------------------------------------------------------------------- random small batches

def test_random_ragged_batches_match_brute_force_and_invariants():
    """Seeded random tiny ragged batches (mixed decode / chunk / empty sequences, GQA groups 1-3,
    block sizes 4 and 8): the vectorised oracle equals the explicit loops, the ragged batch
    equals each sequence run alone, and every output lies in the hull of its visible values."""
    rng = np.random.default_rng(2024)
    for trial in range(12):
        S = int(rng.integers(1, 4))
        G = int(rng.integers(1, 4))
        Hkv = int(rng.integers(1, 3))
        bs = int(rng.choice([4, 8]))
        q_lens = [int(rng.choice([0, 1, 1, int(rng.integers(2, 6))])) for _ in range(S)]
        kv_lens = [q + int(rng.integers(0, 10)) for q in q_lens]
        kv_lens = [max(k, 1) if q == 0 else k for q, k in zip(q_lens, kv_lens)]
        b = workloads.build_batch(q_lens, kv_lens, G * Hkv, Hkv, 4, bs, seed=700 + trial)
        kp, vp = _appended(b)
        out, lse = _attend(b, kp, vp)
        ref = _brute_force(_f64(b.q).tolist(), _f64(kp).tolist(), _f64(vp).tolist(),
                           b.block_table.tolist(), b.cu_seqlens_q.tolist(), b.kv_lens.tolist(),
                           bs, b.scale)
        assert np.allclose(out, ref, rtol=0, atol=1e-12), trial
        for s in range(S):
            a, e = int(b.cu_seqlens_q[s]), int(b.cu_seqlens_q[s + 1])
            o1, l1 = opa.ragged_paged_attention(b.q[a:e], kp, vp, b.block_table[s:s + 1],
                                                [0, e - a], b.kv_lens[s:s + 1], bs, b.scale)
            assert np.array_equal(o1, out[a:e]) and np.array_equal(l1, lse[a:e]), trial
            ctx = int(b.kv_lens[s]) - (e - a)
            for i in range(e - a):
                keys = np.arange(ctx + i + 1)
                rows = b.block_table[s][keys // bs] * bs + keys % bs
                vis = _f64(vp).reshape(-1, Hkv, 4)[rows]            # [keys, Hkv, D]
                for h in range(G * Hkv):
                    v = vis[:, h // G, :]
                    o = out[a + i, h]
                    assert np.all(o >= v.min(0) - 1e-12) and np.all(o <= v.max(0) + 1e-12), trial
