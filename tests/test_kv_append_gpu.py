"""KV-append through the C ABI: the whole page pool must match the oracle bit for bit."""
import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from gpu_util import DeviceBatch, named_config, bits_of, i32, oracle_append

pytestmark = pytest.mark.gpu


def _check_pool(db, b):
    k_ref, v_ref = oracle_append(b)
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    assert np.array_equal(bits_of(db.k_pages), k_ref)
    assert np.array_equal(bits_of(db.v_pages), v_ref)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_append_configs_bit_exact(cuda_lib, cfg):
    b = named_config(cfg)
    _check_pool(DeviceBatch(b), b)


@pytest.mark.parametrize("bs", [4, 16, 32, 64, 256])
@pytest.mark.parametrize("D", [64, 128])
def test_append_ragged_small(cuda_lib, bs, D):
    # ragged mix: decodes, chunks crossing block boundaries, an empty sequence, a full table
    q_lens = [1, 37, 0, 5, 1, 130]
    kv_lens = [1, 37, 9, 70, 2 * bs, 300]
    b = workloads.build_batch(q_lens, kv_lens, 8, 4, D, bs, seed=40 + bs + D)
    _check_pool(DeviceBatch(b), b)


@pytest.mark.parametrize("Hkv", [1, 3, 32])
def test_append_row_widths(cuda_lib, Hkv):
    # a token row of Hkv * D bf16: narrower than one 16-byte chunk per lane (Hkv 1, D 64),
    # not a multiple of the warp (Hkv 3), and wider than one pass of the warp (Hkv 32, D 128)
    D = 64 if Hkv == 1 else 128
    q_lens = [1, 70, 3, 1]
    kv_lens = [40, 70, 19, 1]
    b = workloads.build_batch(q_lens, kv_lens, Hkv, Hkv, D, 16, seed=60 + Hkv)
    _check_pool(DeviceBatch(b), b)


def test_append_many_sequences(cuda_lib):
    # 3000 sequences: several rounds of the warp's 32-way search for a token's sequence
    rng = np.random.default_rng(61)
    q_lens = [int(x) for x in rng.integers(0, 4, 3000)]
    kv_lens = [q + int(rng.integers(0, 40)) for q in q_lens]
    b = workloads.build_batch(q_lens, kv_lens, 4, 2, 64, 16, seed=62)
    _check_pool(DeviceBatch(b), b)


def test_append_max_table_and_idempotent(cuda_lib):
    bs = 16
    b = workloads.build_batch([3, 1], [64, 64], 4, 2, 128, bs, seed=7, max_blocks=4)  # full tables
    db = DeviceBatch(b)
    _check_pool(db, b)
    before = bits_of(db.k_pages).copy()
    db.append()  # same step again: same slots, same bits
    assert np.array_equal(bits_of(db.k_pages), before)


def test_append_empty_batch_is_noop(cuda_lib):
    b = workloads.build_batch([0, 0], [5, 9], 4, 2, 64, 16, seed=3)
    db = DeviceBatch(b)
    before = bits_of(db.k_pages).copy()
    db.append()
    assert cb.get_device_error() == cb.CB_OK
    assert np.array_equal(bits_of(db.k_pages), before)


def test_append_bad_block_id_is_reported_and_skipped(cuda_lib):
    b = workloads.build_batch([2, 1], [20, 5], 4, 2, 64, 16, seed=5)
    db = DeviceBatch(b)
    table = b.block_table.copy()
    table[0, 1] = b.num_pages + 3          # positions 18, 19 of sequence 0 now point outside
    db.block_table = i32(table)
    before_k = bits_of(db.k_pages).copy()
    db.append()
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    assert cb.get_device_error() == cb.CB_OK          # reading clears the word
    after_k = bits_of(db.k_pages)
    # only sequence 1's token (position 4, block table[1][0], offset 4) was written
    changed = np.argwhere(np.any(after_k != before_k, axis=(2, 3)))
    assert changed.tolist() == [[int(table[1, 0]), 4]]


def test_append_kv_shorter_than_q_is_reported(cuda_lib):
    b = workloads.build_batch([3], [8], 4, 2, 64, 16, seed=6)
    db = DeviceBatch(b)
    db.kv_lens = i32([2])
    before = bits_of(db.k_pages).copy()
    db.append()
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    assert np.array_equal(bits_of(db.k_pages), before)
