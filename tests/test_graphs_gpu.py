"""The append + attention pass replayed from CUDA graphs (continuous_batching_paged_gb300.graphs)
gives bit-for-bit the outputs and page pools of the eager calls, over batches of changing
shapes; and padding rows past cu_seqlens_q[S] are neither read nor written."""
import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
from continuous_batching_paged_gb300.graphs import GraphedStep
from gpu_util import assert_close, bf16_tensor, bits_of, i32, oracle_append
from oracle import paged_attention as opa
import workloads

pytestmark = pytest.mark.gpu


def _steps():
    # (q_lens, kv_lens) of successive batches; some share a padded shape (replays)
    return [
        ([1] * 5, [40, 300, 17, 1000, 65]),
        ([1] * 7, [41, 301, 18, 1001, 66, 3, 129]),          # same bucket as the first
        ([1, 1, 130, 1], [42, 302, 130 + 20, 1002]),
        ([64, 1, 1], [64, 303, 19]),
        ([1] * 20, list(range(30, 50))),                     # a second sequence bucket
        ([1, 1, 130, 1], [43, 303, 130 + 21, 1003]),          # first chunk bucket again
    ]


def _batch(q_lens, kv_lens, seed):
    return workloads.build_batch(q_lens, kv_lens, 8, 2, 128, 16, seed=seed, num_pages=400,
                                 max_blocks=80, shuffle_pages=True, name="graph step")


def test_graph_replay_matches_eager_bit_for_bit(cuda_lib):
    b0 = _batch(*_steps()[0], seed=500)
    kp_e, vp_e = bf16_tensor(b0.k_pages), bf16_tensor(b0.v_pages)
    kp_g, vp_g = kp_e.clone(), vp_e.clone()
    g = GraphedStep(kp_g, vp_g, 16, b0.scale, 8, 80, seq_interval=8, token_interval=64)
    for i, (ql, kl) in enumerate(_steps()):
        b = _batch(ql, kl, seed=500 + i)
        kp_e.copy_(bf16_tensor(b.k_pages))       # this step's cache content, in place
        vp_e.copy_(bf16_tensor(b.v_pages))
        kp_g.copy_(kp_e)
        vp_g.copy_(vp_e)
        q, kn, vn = bf16_tensor(b.q), bf16_tensor(b.k_new), bf16_tensor(b.v_new)
        tab, cu, kv = i32(b.block_table), i32(b.cu_seqlens_q), i32(b.kv_lens)
        cb.kv_append(kn, vn, kp_e, vp_e, tab, cu, kv, 16)
        out_e = cb.ragged_paged_attention(q, kp_e, vp_e, tab, cu, kv, 16, b.scale)
        out_g = g.run(q, kn, vn, tab, cu, kv)
        assert cb.get_device_error() == cb.CB_OK
        assert torch.equal(out_e.view(torch.int16), out_g.view(torch.int16)), f"step {i}"
        assert torch.equal(kp_e.view(torch.int16), kp_g.view(torch.int16))
        assert torch.equal(vp_e.view(torch.int16), vp_g.view(torch.int16))
        if i == 2:
            k_ref, v_ref = oracle_append(b)
            ref, _ = opa.ragged_paged_attention(b.q, k_ref, v_ref, b.block_table,
                                                b.cu_seqlens_q, b.kv_lens, 16, b.scale)
            assert_close(out_g.float().cpu().numpy(), ref, "graph replay vs oracle")
    # buckets: (8, 64) x2, (8, 192) x2, (8, 128), (24, 64): four captures for six steps
    assert g.captures == 4


def test_graph_cache_evicts_least_recently_used(cuda_lib):
    b = _batch([1, 1], [40, 50], seed=520)
    kp, vp = bf16_tensor(b.k_pages), bf16_tensor(b.v_pages)
    g = GraphedStep(kp, vp, 16, b.scale, 8, 80, seq_interval=4, token_interval=64, max_graphs=1)
    args = lambda bb: (bf16_tensor(bb.q), bf16_tensor(bb.k_new), bf16_tensor(bb.v_new),
                       i32(bb.block_table), i32(bb.cu_seqlens_q), i32(bb.kv_lens))
    small, large = _batch([1, 1], [40, 50], 521), _batch([1] * 6, [40] * 6, 522)
    for bb in (small, small, large, small):
        g.run(*args(bb))
    assert g.captures == 3 and len(g.cache) == 1


def test_padding_rows_are_neither_read_nor_written(cuda_lib):
    b = _batch([1, 3, 1], [40, 70, 9], seed=530)
    T, pad = b.num_tokens, 11
    rng = np.random.default_rng(531)
    junk = lambda shape: workloads.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    q = bf16_tensor(np.concatenate([b.q, junk((pad,) + b.q.shape[1:])]))
    kn = bf16_tensor(np.concatenate([b.k_new, junk((pad,) + b.k_new.shape[1:])]))
    vn = bf16_tensor(np.concatenate([b.v_new, junk((pad,) + b.v_new.shape[1:])]))
    kp, vp = bf16_tensor(b.k_pages), bf16_tensor(b.v_pages)
    tab, cu, kv = i32(b.block_table), i32(b.cu_seqlens_q), i32(b.kv_lens)
    cb.kv_append(kn, vn, kp, vp, tab, cu, kv, 16)
    out = torch.full_like(q, 7.0)
    cb.ragged_paged_attention(q, kp, vp, tab, cu, kv, 16, b.scale, out=out)
    assert cb.get_device_error() == cb.CB_OK
    k_ref, v_ref = oracle_append(b)
    assert np.array_equal(bits_of(kp), k_ref) and np.array_equal(bits_of(vp), v_ref)
    ref, _ = opa.ragged_paged_attention(b.q, k_ref, v_ref, b.block_table, b.cu_seqlens_q,
                                        b.kv_lens, 16, b.scale)
    assert_close(out[:T].float().cpu().numpy(), ref, "rows before the padding")
    assert (out[T:].float() == 7.0).all()
