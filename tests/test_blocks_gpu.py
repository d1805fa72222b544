"""Block moves on the GPU (cb_copy_blocks, cb_kv_offload, cb_kv_restore) bit-exact against the
oracle, and a multi-step continuous-batching loop in which the native scheduler's batches
(including copy-on-write block copies of forked requests) drive the append and attention
kernels, step by step against the oracle."""
import random

import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
from continuous_batching_paged_gb300.runtime import BlockAllocator, Scheduler
from gpu_util import assert_close, bf16_tensor, bits_of, i32
from oracle import blocks as ob
from oracle import paged_attention as opa
import workloads

pytestmark = pytest.mark.gpu


def _pools(P, bs, H, D, seed):
    rng = np.random.default_rng(seed)
    k = workloads.f32_to_bf16_bits(rng.standard_normal((P, bs, H, D), dtype=np.float32))
    v = workloads.f32_to_bf16_bits(rng.standard_normal((P, bs, H, D), dtype=np.float32))
    return k, v


@pytest.mark.parametrize("bs,H,D", [(4, 1, 64), (16, 8, 128), (64, 2, 64), (32, 8, 128)])
def test_copy_blocks_bit_exact(cuda_lib, bs, H, D):
    P = 97
    k, v = _pools(P, bs, H, D, seed=bs + H + D)
    rng = np.random.default_rng(7)
    perm = rng.permutation(P)
    src, dst = perm[:30], perm[30:60]                     # disjoint: no block read and written
    src = np.concatenate([src, [perm[70]]])
    dst = np.concatenate([dst, [perm[70]]])               # a src == dst pair: no-op
    kp, vp = bf16_tensor(k), bf16_tensor(v)
    cb.copy_blocks(kp, vp, i32(src), i32(dst), bs)
    assert cb.get_device_error() == cb.CB_OK
    assert np.array_equal(bits_of(kp), ob.copy_blocks(k, src, dst))
    assert np.array_equal(bits_of(vp), ob.copy_blocks(v, src, dst))


def test_copy_blocks_bad_id_reported_and_skipped(cuda_lib):
    P, bs, H, D = 20, 16, 2, 64
    k, v = _pools(P, bs, H, D, seed=3)
    kp, vp = bf16_tensor(k), bf16_tensor(v)
    cb.copy_blocks(kp, vp, i32([1, 2, 3]), i32([5, P + 4, 6]), bs)
    assert cb.get_device_error() == cb.CB_ERR_OUT_OF_RANGE
    assert np.array_equal(bits_of(kp), ob.copy_blocks(k, [1, 3], [5, 6]))
    cb.copy_blocks(kp, vp, i32([0]), i32([9]), bs)         # the context is still usable
    assert cb.get_device_error() == cb.CB_OK


@pytest.mark.parametrize("bs,H,D", [(16, 8, 128), (4, 2, 64)])
def test_offload_restore_bit_exact(cuda_lib, bs, H, D):
    P = 300
    k, v = _pools(P, bs, H, D, seed=11)
    kp, vp = bf16_tensor(k), bf16_tensor(v)
    rng = np.random.default_rng(12)
    blocks = rng.permutation(P)[:77]
    hk = torch.empty((77, bs, H, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((77, bs, H, D), dtype=torch.bfloat16).pin_memory()
    cb.kv_offload(kp, vp, i32(blocks), bs, hk, hv)
    torch.cuda.synchronize()
    assert cb.get_device_error() == cb.CB_OK
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), ob.gather_blocks(k, blocks))
    assert np.array_equal(hv.view(torch.int16).numpy().view(np.uint16), ob.gather_blocks(v, blocks))
    # restore into other blocks
    others = np.setdiff1d(np.arange(P), blocks)[:77]
    cb.kv_restore(kp, vp, i32(others), bs, hk, hv)
    assert cb.get_device_error() == cb.CB_OK
    host_k = ob.gather_blocks(k, blocks)
    assert np.array_equal(bits_of(kp), ob.scatter_blocks(k, others, host_k))
    assert np.array_equal(bits_of(vp), ob.scatter_blocks(v, others, ob.gather_blocks(v, blocks)))


@pytest.mark.parametrize("policy", ["fifo", "prefill_first"])
def test_scheduler_driven_steps_match_oracle(cuda_lib, policy):
    # A continuous-batching loop: the native scheduler builds each step (decodes, prefill
    # chunks, forks with copy-on-write), the GPU copies the blocks, appends and attends; the
    # oracle replays the same steps on its own pools.
    P, bs, Hq, Hkv, D, MB = 400, 16, 8, 2, 64, 24
    rng = random.Random(17)
    nrng = np.random.default_rng(18)
    alloc = BlockAllocator(P, bs, MB)
    sched = Scheduler(alloc, max_batch_tokens=96, max_requests_per_batch=8, policy=policy)
    for r in range(12):
        sched.add_request(r, rng.randint(1, 150), rng.randint(2, 14))
    k_or, v_or = _pools(P, bs, Hkv, D, seed=19)
    kp, vp = bf16_tensor(k_or), bf16_tensor(v_or)
    next_id, steps, copies = 100, 0, 0
    scale = 1.0 / np.sqrt(D)
    while sched.num_active():
        step = sched.step()
        steps += 1
        assert steps < 500
        S = len(step["seq_ids"])
        if S:
            src, dst = step["cow_src"].copy(), step["cow_dst"].copy()
            if len(src):
                copies += len(src)
                cb.copy_blocks(kp, vp, i32(src), i32(dst), bs)
                k_or, v_or = ob.copy_blocks(k_or, src, dst), ob.copy_blocks(v_or, src, dst)
            T = int(step["num_tokens"])
            draw = lambda *shape: workloads.f32_to_bf16_bits(
                nrng.standard_normal(shape, dtype=np.float32))
            q, kn, vn = draw(T, Hq, D), draw(T, Hkv, D), draw(T, Hkv, D)
            table = step["block_table"].copy()
            cu, kvl = step["cu_seqlens_q"].copy(), step["kv_lens"].copy()
            cb.kv_append(bf16_tensor(kn), bf16_tensor(vn), kp, vp, i32(table), i32(cu), i32(kvl), bs)
            out = cb.ragged_paged_attention(bf16_tensor(q), kp, vp, i32(table), i32(cu), i32(kvl),
                                            bs, scale)
            assert cb.get_device_error() == cb.CB_OK
            k_or, v_or = opa.kv_append(kn, vn, k_or, v_or, table, cu, kvl, bs)
            ref, _ = opa.ragged_paged_attention(q, k_or, v_or, table, cu, kvl, bs, scale)
            assert_close(out.float().cpu().numpy(), ref, f"step {steps}")
        # fork a decoding request now and then (parallel sampling)
        if steps % 4 == 2:
            ids = [int(x) for x, ql in zip(step["seq_ids"], np.diff(step["cu_seqlens_q"])) if ql == 1]
            if ids:
                try:
                    sched.fork_request(ids[0], next_id, rng.randint(3, 14))
                    next_id += 1
                except cb.CbError:
                    pass   # parent already at its last token
    assert copies > 0
    assert np.array_equal(bits_of(kp), k_or) and np.array_equal(bits_of(vp), v_or)


def _rows(seed, shape):
    rng = np.random.default_rng(seed)
    return workloads.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _prefix_run(prefix, requests, P, bs, Hq, Hkv, D, MB):
    """Run `requests` (id, tokens, new) through the native scheduler and the GPU path; every
    token's q/k/v rows are a function of its request's token prefix (prompt positions) or of
    (request, position) (generated positions), as a model's would be.  Returns the output row
    of every computed (request, position) and checks each step against the oracle."""
    alloc = BlockAllocator(P, bs, MB)
    alloc.set_prefix_caching(prefix)
    sched = Scheduler(alloc, max_batch_tokens=80, max_requests_per_batch=6)
    seeds = {}
    for rid, toks, new in requests:
        sched.add_request_tokens(rid, toks, new)
        h, hs = 0, []
        for t in toks:
            h = (h * 1000003 + t + 1) % (1 << 61)
            hs.append(h)
        seeds[rid] = hs
    k_or = np.zeros((P, bs, Hkv, D), dtype=np.uint16)
    v_or = np.zeros_like(k_or)
    kp, vp = bf16_tensor(k_or), bf16_tensor(v_or)
    scale = 1.0 / np.sqrt(D)
    outs, cached, steps = {}, 0, 0
    while sched.num_active():
        st = sched.step()
        steps += 1
        assert steps < 400
        cached += st["num_cached"]
        S = len(st["seq_ids"])
        if S == 0:
            continue
        cu, kvl, table = (st["cu_seqlens_q"].copy(), st["kv_lens"].copy(),
                          st["block_table"].copy())
        qs, ks, vs, keys = [], [], [], []
        for i, rid in enumerate(st["seq_ids"].tolist()):
            n = int(cu[i + 1] - cu[i])
            for p in range(int(kvl[i]) - n, int(kvl[i])):
                hs = seeds[rid]
                sd = hs[p] if p < len(hs) else (rid * 1000003 + p) * 7 + 5
                qs.append(_rows(sd * 3 + 0, (Hq, D)))
                ks.append(_rows(sd * 3 + 1, (Hkv, D)))
                vs.append(_rows(sd * 3 + 2, (Hkv, D)))
                keys.append((rid, p))
        q, kn, vn = np.stack(qs), np.stack(ks), np.stack(vs)
        cb.kv_append(bf16_tensor(kn), bf16_tensor(vn), kp, vp, i32(table), i32(cu), i32(kvl), bs)
        out = cb.ragged_paged_attention(bf16_tensor(q), kp, vp, i32(table), i32(cu), i32(kvl),
                                        bs, scale).float().cpu().numpy()
        assert cb.get_device_error() == cb.CB_OK
        k_or, v_or = opa.kv_append(kn, vn, k_or, v_or, table, cu, kvl, bs)
        ref, _ = opa.ragged_paged_attention(q, k_or, v_or, table, cu, kvl, bs, scale)
        assert_close(out, ref, f"prefix={prefix} step {steps}")
        for j, key in enumerate(keys):
            outs[key] = out[j]
    return outs, cached


def test_prefix_cache_gives_the_outputs_of_a_full_prefill(cuda_lib):
    # requests sharing system prompts: with the prefix cache on, later requests skip the
    # cached blocks' prefill, and every row they do compute equals the row computed with the
    # cache off (each position's K/V is a function of its token prefix, as a model's would be)
    rng = random.Random(23)
    systems = [[rng.randrange(30000) for _ in range(n)] for n in (150, 90)]
    requests = []
    for rid in range(10):
        sysp = systems[rid % 2][:rng.randint(40, 150)]
        toks = sysp + [rng.randrange(30000) for _ in range(rng.randint(1, 40))]
        requests.append((rid, toks, rng.randint(1, 6)))
    P, bs, Hq, Hkv, D, MB = 200, 16, 8, 2, 64, 16
    full, c0 = _prefix_run(False, requests, P, bs, Hq, Hkv, D, MB)
    hit, c1 = _prefix_run(True, requests, P, bs, Hq, Hkv, D, MB)
    assert c0 == 0 and c1 > 0
    assert set(hit) <= set(full) and len(hit) < len(full)
    for key, row in hit.items():
        assert_close(row, full[key].astype(np.float64), f"row {key}", atol=4e-2, rtol=2e-2)
