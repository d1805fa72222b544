"""Device-side checks of bad metadata, and the chunk pass's block-table reads past its
shared-memory copy of the table row.

Bad metadata is reported through the device error word (CB_ERR_OUT_OF_RANGE) and never traps:
the kernels skip what the check guards.  Each batch below is built so that even an access the
check failed to guard would stay inside the allocated buffers (the bad sequence sits in an inner
row of the block table, so a read past its row lands in the next row; the token tensors carry
rows past num_tokens), which makes a missing check show up as a wrong value instead of a fault.
The valid sequences must still give the oracle's result, and nothing outside the slots the valid
metadata names may change.
"""
import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from gpu_util import DeviceBatch, assert_close, bf16_tensor, bits_of, i32, oracle_append
from oracle import paged_attention as opa

pytestmark = pytest.mark.gpu


def _expected_pool(b, pages, new, tokens):
    """The original pool with only the listed (sequence, query index) rows appended, by the
    slot rule of the oracle."""
    exp = np.array(pages, copy=True)
    flat = exp.reshape(b.num_pages * b.block_size, b.num_kv_heads, b.head_dim)
    q_lens = np.diff(b.cu_seqlens_q)
    for s, i in tokens:
        pos = int(b.kv_lens[s]) - int(q_lens[s]) + i
        flat[opa.slot_of(b.block_table[s], pos, b.block_size, b.num_pages)] = new[int(b.cu_seqlens_q[s]) + i]
    return exp


def _attend_padded(db, cu, kv_lens=None, T=None, pad=8):
    """Attention with the given metadata; q and out are views of buffers `pad` rows longer, so
    a stray access past num_tokens stays in memory the test can inspect."""
    b = db.b
    T = b.num_tokens if T is None else T
    q_full = torch.zeros((T + pad, b.num_q_heads, b.head_dim), dtype=torch.bfloat16, device="cuda")
    q_full[:b.num_tokens] = db.q[:T] if T <= b.num_tokens else db.q
    out_full = torch.full_like(q_full, 7.0)
    cb.ragged_paged_attention(q_full[:T], db.k_pages, db.v_pages, db.block_table, i32(cu),
                              db.kv_lens if kv_lens is None else i32(kv_lens), b.block_size,
                              b.scale, out=out_full[:T])
    return out_full, cb.get_device_error()


def _reference_rows(b, kp, vp, seqs):
    ref, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                        b.block_size, b.scale)
    rows = [int(b.cu_seqlens_q[s]) for s in seqs]
    return rows, ref[rows]


# ------------------------------------------------------------------ chunk block-table fallback

@pytest.mark.parametrize("bs,ctx,q_len,G", [(4, 4300, 200, 1), (4, 4400, 130, 4),
                                            (16, 16600, 130, 4), (16, 16550, 257, 1)])
def test_chunk_reads_table_entries_past_its_shared_copy(cuda_lib, bs, ctx, q_len, G):
    # one chunk whose block-table row holds more entries than the chunk pass stages in shared
    # memory (a prior context of 4300 tokens at block size 4 is 1075+ entries; 16600 at block
    # size 16, 1038+), so its later K/V tiles take the entries from global memory; a decode
    # token and a short chunk ride along
    b = workloads.build_batch([1, q_len, 3], [700, ctx + q_len, 90], 2 * G, 2, 128, bs,
                              seed=950 + bs + G, name=f"long table bs{bs}")
    db = DeviceBatch(b)
    db.append()
    out, lse = db.attend(lse=True)
    assert cb.get_device_error() == cb.CB_OK
    kp, vp = oracle_append(b)
    ref, ref_lse = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q,
                                              b.kv_lens, b.block_size, b.scale)
    assert_close(out.float().cpu().numpy(), ref, b.name)
    assert_close(lse.cpu().numpy(), ref_lse, b.name + " lse", atol=1e-3, rtol=1e-3)


# ------------------------------------------------------------------ malformed cu_seqlens_q

def _malformed_batch():
    # decodes and chunks; sequence 3 is a decode with a short context so that a token range
    # that grows into it fails kv_len >= q_len
    q_lens = [1, 40, 1, 1, 60, 1]
    kv_lens = [300, 240, 77, 5, 160, 1000]
    return workloads.build_batch(q_lens, kv_lens, 8, 2, 128, 16, seed=961, name="malformed")


def test_decreasing_cu_seqlens_reported(cuda_lib):
    b = _malformed_batch()
    cu_bad = b.cu_seqlens_q.copy()
    assert list(cu_bad) == [0, 1, 41, 42, 43, 103, 104]
    cu_bad[3] = 30            # sequence 2: [41, 30), sequence 3: [30, 43)
    kp, vp = oracle_append(b)

    # attention on correctly appended pages: the error is reported, the chunk pass is given
    # no work, the valid decode sequences 0 and 5 are exact, nothing past num_tokens changes
    db = DeviceBatch(b)
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    out_full, st = _attend_padded(db, cu_bad)
    assert st == cb.CB_ERR_OUT_OF_RANGE
    rows, ref = _reference_rows(b, kp, vp, [0, 5])
    assert_close(out_full[rows].float().cpu().numpy(), ref, "valid decodes beside a bad cu")
    assert bool((out_full[b.num_tokens:] == 7.0).all())

    # the stand-alone append: reported; tokens of well-formed ranges land where they belong;
    # the rest of the pool either keeps its bits or holds the row the valid metadata puts there
    for fused in (False, True):
        db = DeviceBatch(b)
        if fused:
            cb.append_attention(db.q, db.k_new, db.v_new, db.k_pages, db.v_pages, db.block_table,
                                i32(cu_bad), db.kv_lens, b.block_size, b.scale)
        else:
            cb.kv_append(db.k_new, db.v_new, db.k_pages, db.v_pages, db.block_table, i32(cu_bad),
                         db.kv_lens, b.block_size)
        assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
        got_k, got_v = bits_of(db.k_pages), bits_of(db.v_pages)
        must = [(0, 0), (4, 0), (5, 0)] + [(1, i) for i in range(29)] + [(4, i) for i in range(60)]
        exp_k = _expected_pool(b, b.k_pages, b.k_new, must)
        exp_v = _expected_pool(b, b.v_pages, b.v_new, must)
        for got, exp, full in ((got_k, exp_k, kp), (got_v, exp_v, vp)):
            diff = got != exp
            # every other change is a valid-metadata row of sequence 1 (its ambiguous tokens)
            assert np.array_equal(got[diff], full[diff])
            must_idx = _expected_pool(b, np.zeros_like(b.k_pages), np.ones_like(b.k_new), must) != 0
            assert np.array_equal(got[must_idx], full[must_idx])


def test_cu_seqlens_past_num_tokens_reported(cuda_lib):
    # cu[S] > T: the last sequence's range runs past the token rows; it is skipped by the
    # append and the planner, the other decodes are exact, no row past T changes
    b = workloads.build_batch([1, 1, 50, 1], [64, 129, 300, 77], 8, 2, 128, 16, seed=963,
                              name="cu past T")
    T = b.num_tokens              # 53
    cu_bad = b.cu_seqlens_q.copy()
    cu_bad[4] = T + 7
    kp, vp = oracle_append(b)
    # k_new / v_new with 8 extra rows of real values past T
    kn = bf16_tensor(np.concatenate([b.k_new, b.k_new[:8]]))[:T]
    vn = bf16_tensor(np.concatenate([b.v_new, b.v_new[:8]]))[:T]
    db = DeviceBatch(b)
    cb.kv_append(kn, vn, db.k_pages, db.v_pages, db.block_table, i32(cu_bad), db.kv_lens,
                 b.block_size)
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    must = [(0, 0), (1, 0)] + [(2, i) for i in range(50)]
    assert np.array_equal(bits_of(db.k_pages), _expected_pool(b, b.k_pages, b.k_new, must))
    assert np.array_equal(bits_of(db.v_pages), _expected_pool(b, b.v_pages, b.v_new, must))

    db = DeviceBatch(b)
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    out_full, st = _attend_padded(db, cu_bad)
    assert st == cb.CB_ERR_OUT_OF_RANGE
    rows, ref = _reference_rows(b, kp, vp, [0, 1])
    assert_close(out_full[rows].float().cpu().numpy(), ref, "valid decodes beside cu[S] > T")
    assert bool((out_full[T:] == 7.0).all())


def test_kv_len_past_table_width_reported(cuda_lib):
    # sequence 1 (an inner row) claims one key more than its table row can name: its appended
    # token would sit in logical block MB, and a read past the row would find row 2's first
    # block (valid), so a missing check would corrupt sequence 2
    bs, MB = 16, 12
    b = workloads.build_batch([1, 1, 1, 1], [100, MB * bs, 150, 33], 8, 2, 128, bs, seed=967,
                              max_blocks=MB, name="table width")
    kv_bad = b.kv_lens.copy()
    kv_bad[1] = MB * bs + 1
    kp, vp = oracle_append(b)
    db = DeviceBatch(b)
    cb.kv_append(db.k_new, db.v_new, db.k_pages, db.v_pages, db.block_table, db.cu, i32(kv_bad),
                 b.block_size)
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    must = [(0, 0), (2, 0), (3, 0)]
    assert np.array_equal(bits_of(db.k_pages), _expected_pool(b, b.k_pages, b.k_new, must))
    assert np.array_equal(bits_of(db.v_pages), _expected_pool(b, b.v_pages, b.v_new, must))

    db = DeviceBatch(b)
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    out_full, st = _attend_padded(db, b.cu_seqlens_q, kv_lens=kv_bad)
    assert st == cb.CB_ERR_OUT_OF_RANGE
    rows, ref = _reference_rows(b, kp, vp, [0, 2, 3])
    assert_close(out_full[rows].float().cpu().numpy(), ref, "valid decodes beside a long kv_len")
    assert bool((out_full[b.num_tokens:] == 7.0).all())
