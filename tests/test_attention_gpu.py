"""Ragged paged attention through the C ABI against the float64 oracle.

Bar: every output element within 2e-2 + 1e-2 * |ref| (bf16 inputs, fp32 accumulation, bf16
output); the softmax normaliser (lse) within 1e-3 + 1e-3 * |ref|; page permutation and prefix
sharing give bit-identical GPU output (the kernels' split points depend only on lengths).
"""
import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from gpu_util import DeviceBatch, named_config, assert_close, bits_of, bf16_tensor, i32, oracle_append
from oracle import paged_attention as opa

pytestmark = pytest.mark.gpu


def _run_full(b, decode_ctas=0):
    """Append on the GPU, attend on the GPU, and compare every element with the oracle."""
    db = DeviceBatch(b)
    db.append()
    out, lse = db.attend(lse=True, decode_ctas=decode_ctas)
    assert cb.get_device_error() == cb.CB_OK
    kp, vp = oracle_append(b)
    ref, ref_lse = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q,
                                              b.kv_lens, b.block_size, b.scale)
    gpu = out.float().cpu().numpy()
    assert_close(gpu, ref, b.name)
    assert_close(lse.cpu().numpy(), ref_lse, b.name + " lse", atol=1e-3, rtol=1e-3)
    return db, out


# ----------------------------------------------------------------------------- small, exhaustive

def test_config1_tiny_ragged(cuda_lib):
    _run_full(named_config(1))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [4, 16, 32, 64, 256])
def test_decode_only_small(cuda_lib, D, bs):
    kv = [1, 2, 15, 16, 17, 100, 257, 1000]
    b = workloads.build_batch([1] * len(kv), kv, 8, 2, D, bs, seed=100 + bs + D,
                              name=f"decode D{D} bs{bs}")
    _run_full(b)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [4, 16, 64, 256])
def test_chunks_small(cuda_lib, D, bs):
    # chunks: ragged tails (130 = 128 + 2), prior context crossing tiles, a chunk at ctx 0
    q_lens = [130, 2, 64, 257]
    kv_lens = [130, 300, 64 + 77, 257 + 128]
    b = workloads.build_batch(q_lens, kv_lens, 4, 2, D, bs, seed=200 + bs + D,
                              name=f"chunks D{D} bs{bs}")
    _run_full(b)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 16])
def test_mixed_gqa_groups(cuda_lib, G):
    Hkv = 2 if G < 16 else 1
    q_lens = [1, 40, 0, 1, 129, 1]
    kv_lens = [33, 40, 12, 500, 129 + 200, 1]
    b = workloads.build_batch(q_lens, kv_lens, Hkv * G, Hkv, 128, 32, seed=300 + G,
                              name=f"mixed G{G}")
    _run_full(b)


@pytest.mark.parametrize("G", [1, 4])
def test_chunks_of_unequal_cost(cuda_lib, G):
    # many chunk work units whose K/V extents differ (prior context 0 .. 3000, ragged tails):
    # the chunk pass takes them longest first, in an order unrelated to the sequence order;
    # G = 1 pairs two query tiles per CTA, G = 4 pairs two query heads of one KV group
    q_lens = [300, 513, 129, 2, 700, 1, 256]
    kv_lens = [300, 513 + 900, 129 + 3000, 2 + 17, 700 + 2000, 40, 256 + 128]
    b = workloads.build_batch(q_lens, kv_lens, 2 * G, 2, 128, 64, seed=400 + G,
                              name=f"unequal chunks G{G}")
    _run_full(b)


def test_invalid_length_reported_and_chunk_pass_skipped(cuda_lib):
    # kv_len < q_len for the second chunk: reported, no fault, the chunk pass does no work and
    # the valid decode sequence is still computed
    b = workloads.build_batch([1, 40, 60], [70, 120, 90], 8, 2, 128, 16, seed=91)
    db = DeviceBatch(b)
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    kv = b.kv_lens.copy()
    kv[2] = 10
    db.kv_lens = i32(kv)
    out = db.attend()
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    kp, vp = oracle_append(b)
    ref, _ = opa.ragged_paged_attention(b.q[:1], kp, vp, b.block_table[:1], b.cu_seqlens_q[:2],
                                        b.kv_lens[:1], b.block_size, b.scale)
    assert_close(out[:1].float().cpu().numpy(), ref, "decode row beside an invalid chunk")


def test_more_sequences_than_the_planner_keeps_on_chip(cuda_lib):
    # 2100 decode and 2100 chunk sequences: past the 2048 the planner mirrors in shared memory,
    # so its searches read the prefix arrays from the workspace
    rng = np.random.default_rng(93)
    n = 2100
    q_lens = [1] * n + [2] * n
    kv_lens = [int(x) for x in rng.integers(1, 40, n)] + [int(x) for x in rng.integers(2, 40, n)]
    order = rng.permutation(2 * n)
    q_lens = [q_lens[i] for i in order]
    kv_lens = [kv_lens[i] for i in order]
    b = workloads.build_batch(q_lens, kv_lens, 4, 2, 64, 16, seed=94, name="4200 seqs")
    _run_full(b)


@pytest.mark.parametrize("G,Hkv,ctas", [(12, 4, 0), (16, 8, 0), (16, 8, 3), (16, 2, 64), (9, 8, 0)])
def test_wide_gqa_groups(cuda_lib, G, Hkv, ctas):
    # more than 8 query heads per KV head: two decode warps share each KV head's query heads
    # (4 KV heads per decode CTA, so Hkv = 8 is two head groups); split and whole decode
    # sequences and a chunk
    q_lens = [1, 1, 1, 1, 1, 130]
    kv_lens = [3000, 17, 800, 4096, 1, 130 + 300]
    b = workloads.build_batch(q_lens, kv_lens, G * Hkv, Hkv, 128, 32, seed=700 + G + Hkv,
                              name=f"G{G} Hkv{Hkv}")
    _run_full(b, decode_ctas=ctas)


def test_many_kv_heads_two_head_groups(cuda_lib):
    b = workloads.build_batch([1, 1, 70], [300, 45, 170], 32, 16, 128, 16, seed=17,
                              name="Hkv16")
    _run_full(b)


@pytest.mark.parametrize("ctas", [1, 3, 64, 512])
def test_decode_split_counts_agree(cuda_lib, ctas):
    kv = [3000, 17, 800, 4096, 1]
    b = workloads.build_batch([1] * 5, kv, 32, 8, 128, 32, seed=23, name=f"splits{ctas}")
    _run_full(b, decode_ctas=ctas)


def test_max_table_length(cuda_lib):
    bs = 64
    mb = 40
    b = workloads.build_batch([1, 200], [mb * bs, mb * bs], 16, 8, 128, bs, seed=31,
                              max_blocks=mb, name="full table")
    _run_full(b)


def test_large_k_scale_softmax_range(cuda_lib):
    b = workloads.build_batch([1, 300], [900, 1300], 8, 2, 128, 64, seed=41, k_scale=4.0,
                              name="K x4")
    _run_full(b)


# ----------------------------------------------------------------------------- invariants

def test_page_permutation_bit_identical(cuda_lib):
    b = workloads.build_batch([1, 77, 1, 3], [400, 300, 64, 129], 8, 2, 128, 16, seed=51)
    db, out = _run_full(b)
    perm = np.random.default_rng(9).permutation(b.num_pages)
    kp = torch.empty_like(db.k_pages)
    vp = torch.empty_like(db.v_pages)
    idx = torch.from_numpy(perm).cuda()
    kp[idx] = db.k_pages
    vp[idx] = db.v_pages
    table = np.where(b.block_table >= 0, perm[np.maximum(b.block_table, 0)], -1)
    out2 = db.attend(block_table=i32(table), k_pages=kp, v_pages=vp)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_shared_prefix_bit_identical_to_copies(cuda_lib):
    b = workloads.build_batch([1, 1, 5], [200, 140, 133], 8, 2, 128, 16, seed=61,
                              shared_prefix=([0, 1, 2], 128))
    db, out = _run_full(b)
    n_sh = 128 // 16
    P = b.num_pages
    kp = torch.cat([db.k_pages, torch.zeros((2 * n_sh,) + tuple(db.k_pages.shape[1:]),
                                            dtype=db.k_pages.dtype, device="cuda")])
    vp = torch.cat([db.v_pages, torch.zeros_like(kp[P:])])
    table = b.block_table.copy()
    for r, s in enumerate((1, 2)):
        for j in range(n_sh):
            new = P + r * n_sh + j
            kp[new] = db.k_pages[int(table[s, j])]
            vp[new] = db.v_pages[int(table[s, j])]
            table[s, j] = new
    out2 = db.attend(block_table=i32(table), k_pages=kp, v_pages=vp)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_empty_and_zero_length(cuda_lib):
    b = workloads.build_batch([0, 2, 0], [5, 9, 0], 4, 2, 64, 16, seed=71)
    _run_full(b)


def test_bad_block_id_reported_without_fault(cuda_lib):
    b = workloads.build_batch([1, 50], [70, 120], 8, 2, 128, 16, seed=81)
    db = DeviceBatch(b)
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    table = b.block_table.copy()
    table[0, 2] = 10 ** 6      # decode sequence
    table[1, 3] = -5           # chunk sequence
    db.attend(block_table=i32(table))
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    # the context is still usable
    out = db.attend()
    assert cb.get_device_error() == cb.CB_OK
    assert torch.isfinite(out.float()).all()


# ----------------------------------------------------------------------------- full-size configs

@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_configs_full_size(cuda_lib, cfg):
    # every element of out and lse of the named full-size batches against the oracle: the
    # decode-only and long-tail batches, the mixed 2048-token batch (a 1928-query chunk at prior
    # context 3000 beside 120 decodes) and the chunk-heavy batch (8 chunks of 512 queries at
    # prior contexts up to 8192, K x4), in the launch configuration the bench times
    b = named_config(cfg)
    db = DeviceBatch(b)
    db.append()
    out, lse = db.attend(lse=True)
    assert cb.get_device_error() == cb.CB_OK
    gpu = out.float().cpu().numpy()
    kp, vp = oracle_append(b)
    assert np.array_equal(bits_of(db.k_pages), kp) and np.array_equal(bits_of(db.v_pages), vp)
    ref, ref_lse = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q,
                                              b.kv_lens, b.block_size, b.scale)
    assert_close(gpu, ref, b.name)
    assert_close(lse.cpu().numpy(), ref_lse, b.name + " lse", atol=1e-3, rtol=1e-3)


# ----------------------------------------------------------------------------- sliding window

@pytest.mark.parametrize("window", [1, 16, 100, 128, 129, 700])
@pytest.mark.parametrize("G", [1, 4])
def test_sliding_window(cuda_lib, window, G):
    # decodes and chunks whose windows start inside, at and across 16-key decode tiles and
    # 128-key chunk tiles; G = 1 pairs query tiles, G = 4 pairs heads
    q_lens = [1, 1, 1, 300, 130, 2, 1]
    kv_lens = [1, 40, 1500, 300 + 900, 130, 2 + 517, 2000]
    b = workloads.build_batch(q_lens, kv_lens, 2 * G, 2, 128, 16, seed=600 + window + G,
                              name=f"window {window} G{G}")
    db = DeviceBatch(b)
    db.append()
    out, lse = cb.ragged_paged_attention(db.q, db.k_pages, db.v_pages, db.block_table, db.cu,
                                         db.kv_lens, b.block_size, b.scale, lse=True,
                                         window=window)
    assert cb.get_device_error() == cb.CB_OK
    kp, vp = oracle_append(b)
    ref, ref_lse = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q,
                                              b.kv_lens, b.block_size, b.scale, window=window)
    assert_close(out.float().cpu().numpy(), ref, f"window {window}")
    assert_close(lse.cpu().numpy(), ref_lse, f"window {window} lse", atol=1e-3, rtol=1e-3)


def test_sliding_window_d64_split_decode(cuda_lib):
    b = workloads.build_batch([1, 1, 64], [3000, 70, 64 + 250], 8, 2, 64, 32, seed=611,
                              name="window D64")
    db = DeviceBatch(b)
    db.append()
    for ctas in (1, 97):
        out = cb.ragged_paged_attention(db.q, db.k_pages, db.v_pages, db.block_table, db.cu,
                                        db.kv_lens, b.block_size, b.scale, window=300,
                                        decode_ctas=ctas)
        assert cb.get_device_error() == cb.CB_OK
        kp, vp = oracle_append(b)
        ref, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q,
                                            b.kv_lens, b.block_size, b.scale, window=300)
        assert_close(out.float().cpu().numpy(), ref, f"window D64 ctas {ctas}")


def test_bounded_wait_times_out_without_fault(cuda_lib):
    # the library's failure path, exercised without a fault: a wait that nothing completes
    # gives up after its limit, the host reads CB_ERR_TIMEOUT, and the context stays usable
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    cb.selftest_wait_timeout(2000, waited)
    assert cb.get_device_error() == cb.CB_ERR_TIMEOUT
    assert 2_000_000 <= int(waited.item()) < 1_000_000_000
    assert cb.get_device_error() == cb.CB_OK          # read and cleared
    _run_full(named_config(1))


@pytest.mark.parametrize("serial", [False, True])
@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_fused_append_attention_equals_separate_calls(cuda_lib, cfg, serial):
    # cb_append_attention (planner overlapping the append) gives the pools and outputs of the
    # two separate calls, bit for bit
    b = named_config(cfg)
    a, f = DeviceBatch(b), DeviceBatch(b)
    a.append()
    out_a = cb.ragged_paged_attention(a.q, a.k_pages, a.v_pages, a.block_table, a.cu,
                                      a.kv_lens, b.block_size, b.scale, serial=serial)
    out_f = cb.append_attention(f.q, f.k_new, f.v_new, f.k_pages, f.v_pages, f.block_table,
                                f.cu, f.kv_lens, b.block_size, b.scale, serial=serial)
    assert cb.get_device_error() == cb.CB_OK
    assert torch.equal(out_a.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(a.k_pages.view(torch.int16), f.k_pages.view(torch.int16))
    assert torch.equal(a.v_pages.view(torch.int16), f.v_pages.view(torch.int16))


@pytest.mark.parametrize("q_lens,kv_lens,has_dec,has_chunk", [
    ([1, 1, 1, 1], [300, 40, 1000, 77], True, False),        # decode tokens only
    ([200, 130], [900, 130], False, True),                   # chunks only
    ([1, 140, 1, 1], [500, 400, 90, 2000], True, True),      # both passes in one launch
])
def test_pass_timestamps_mark_the_passes_that_ran(cuda_lib, q_lens, kv_lens, has_dec, has_chunk):
    # the attention launch stamps the first start and last end of each pass that had work;
    # a pass without work reports (0, 0)
    b = workloads.build_batch(q_lens, kv_lens, 8, 2, 128, 16, seed=77, num_pages=600,
                              max_blocks=160, shuffle_pages=True, name="stamps")
    db = DeviceBatch(b)
    db.append()
    ws = torch.empty(cb.workspace_size(b.num_seqs, 8, 2, 128, b.num_tokens), dtype=torch.uint8,
                     device="cuda")
    out = cb.ragged_paged_attention(db.q, db.k_pages, db.v_pages, db.block_table, db.cu,
                                    db.kv_lens, 16, b.scale, workspace=ws)
    ts = cb.pass_timestamps(ws)
    assert cb.get_device_error() == cb.CB_OK
    assert (ts[0] < ts[1]) == has_dec and (ts[0] == ts[1] == 0) == (not has_dec)
    assert (ts[2] < ts[3]) == has_chunk and (ts[2] == ts[3] == 0) == (not has_chunk)
    kp, vp = oracle_append(b)
    ref, _ = opa.ragged_paged_attention(b.q, kp, vp, b.block_table, b.cu_seqlens_q, b.kv_lens,
                                        16, b.scale)
    assert_close(out.float().cpu().numpy(), ref, "stamps batch")
