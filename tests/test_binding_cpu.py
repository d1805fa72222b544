"""The Python binding on a machine without a GPU: it validates and marshals arguments and
refuses host tensors, so no call can silently compute on the CPU (there is no CPU fallback)."""
import pytest
import torch

import continuous_batching_paged_gb300 as cb


def _host_batch(T=3, S=2, Hq=4, Hkv=2, D=64, P=8, bs=16, MB=4, dtype=torch.bfloat16):
    q = torch.zeros(T, Hq, D, dtype=dtype)
    kp = torch.zeros(P, bs, Hkv, D, dtype=dtype)
    table = torch.zeros(S, MB, dtype=torch.int32)
    cu = torch.tensor([0, 1, T], dtype=torch.int32)
    kv = torch.tensor([5, 2], dtype=torch.int32)
    return q, kp, kp.clone(), table, cu, kv


def test_attention_refuses_host_tensors():
    q, kp, vp, table, cu, kv = _host_batch()
    with pytest.raises(ValueError, match="CUDA tensor"):
        cb.ragged_paged_attention(q, kp, vp, table, cu, kv, 16, 0.125)


def test_append_attention_refuses_host_tensors():
    q, kp, vp, table, cu, kv = _host_batch()
    kn = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cb.append_attention(q, kn, kn.clone(), kp, vp, table, cu, kv, 16, 0.125)


def test_kv_append_refuses_host_tensors():
    q, kp, vp, table, cu, kv = _host_batch()
    kn = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        cb.kv_append(kn, kn.clone(), kp, vp, table, cu, kv, 16)


def test_wrong_dtypes_are_rejected_before_the_library():
    q, kp, vp, table, cu, kv = _host_batch(dtype=torch.float32)
    with pytest.raises(ValueError, match="bfloat16"):
        cb.ragged_paged_attention(q, kp, vp, table, cu, kv, 16, 0.125)


def test_block_moves_refuse_host_tensors():
    _, kp, vp, *_ = _host_batch()
    ids = torch.tensor([0, 1], dtype=torch.int32)
    with pytest.raises(ValueError):
        cb.copy_blocks(kp, vp, ids, ids.flip(0), 16)


def test_graph_buckets_pad_sequences_and_tokens_to_their_intervals():
    from continuous_batching_paged_gb300.graphs import GraphedStep
    pool = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16)
    g = GraphedStep(pool, pool, 16, 0.125, 4, 8, seq_interval=16, token_interval=64)
    assert g.bucket_of(1, 1) == (16, 64)
    assert g.bucket_of(16, 64) == (16, 64)
    assert g.bucket_of(17, 65) == (32, 128)
    assert g.bucket_of(121, 2048) == (128, 2048)
    assert g.captures == 0 and len(g.cache) == 0      # nothing is captured without a device
