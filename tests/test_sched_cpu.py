"""The native allocator and scheduler (libcb host runtime, include/cb_sched.h) against the
Python oracle (oracle/scheduler.py), step by step on seeded random request streams: every
batch must agree exactly (sequence order, query lengths, kv_lens, block tables, copy-on-write
pairs, decode count, retirements), and so must the allocator's free count and reference counts.
No GPU is involved: the library's host runtime makes no CUDA call."""
import random

import numpy as np
import pytest

from continuous_batching_paged_gb300 import CbError
from continuous_batching_paged_gb300.runtime import BlockAllocator, Scheduler
from oracle import scheduler as osch


def _same_step(nb, ob, max_blocks):
    assert nb["seq_ids"].tolist() == ob["seq_ids"]
    assert np.diff(nb["cu_seqlens_q"]).tolist() == ob["q_lens"]
    assert nb["cu_seqlens_q"][0] == 0
    assert nb["kv_lens"].tolist() == ob["kv_lens"]
    for row, table in zip(nb["block_table"], ob["tables"]):
        assert row[:len(table)].tolist() == table
        assert (row[len(table):] == -1).all()
    assert list(zip(nb["cow_src"].tolist(), nb["cow_dst"].tolist())) == ob["copies"]
    assert nb["num_decode"] == ob["num_decode"]
    assert nb["num_finished"] == ob["finished"]
    assert nb["num_tokens"] == sum(ob["q_lens"])


def _drive(seed, policy, num_blocks, bs, max_blocks, budget, cap, n_req, fork_p=0.0,
           arrive_every=3, prefix=False):
    rng = random.Random(seed)
    na = BlockAllocator(num_blocks, bs, max_blocks)
    if prefix:
        na.set_prefix_caching(True)
    ns = Scheduler(na, budget, cap, policy)
    oa = osch.BlockAllocator(num_blocks, bs, max_blocks, prefix_caching=prefix)
    os_ = osch.Scheduler(oa, budget, cap, policy)
    systems = [[rng.randrange(1000) for _ in range(rng.randint(1, 300))] for _ in range(4)]
    pending = []
    for r in range(n_req):
        limit = max_blocks * bs
        if prefix:
            # a shared system prompt (or part of one) and a private suffix
            sysp = rng.choice(systems)[:rng.randint(0, 300)]
            toks = sysp + [rng.randrange(1000) for _ in range(rng.randint(1, 200))]
            toks = toks[:limit - 1]
            p = len(toks)
        else:
            toks = None
            p = rng.randint(1, min(600, limit - 1))
        n = rng.randint(1, min(60, limit - p + 1))
        pending.append((r, p, n, toks))
    next_id = n_req
    steps = 0
    cached_total = [0]
    while pending or os_.num_active():
        # a few arrivals every `arrive_every` steps
        if pending and steps % arrive_every == 0:
            for _ in range(rng.randint(1, 4)):
                if pending:
                    r, p, n, toks = pending.pop(0)
                    if toks is None:
                        ns.add_request(r, p, n)
                    else:
                        ns.add_request_tokens(r, toks, n)
                    os_.add_request(r, p, n, toks)
        # parallel sampling: fork a decoding request now and then
        if fork_p and rng.random() < fork_p:
            dec = [q for q in os_.requests if q.state == osch.DECODE and q.generated < q.max_new]
            if dec:
                par = rng.choice(dec)
                limit = (max_blocks * bs) - par.prompt + 1
                mx = rng.randint(par.generated, max(par.generated, min(limit, par.max_new + 10)))
                ns.fork_request(par.id, next_id, mx)
                os_.fork_request(par.id, next_id, mx)
                next_id += 1
        nb, ob = ns.step(), os_.step()
        _same_step(nb, ob, max_blocks)
        assert nb["num_cached"] == ob["cached"]
        cached_total[0] += ob["cached"]
        assert na.num_free() == oa.num_free()
        assert na.num_cached() == len(oa.cache)
        assert [na.ref_count(b) for b in range(num_blocks)] == oa.ref
        steps += 1
        assert steps < 20000
        if not ob["seq_ids"] and not pending and os_.num_active():
            break  # stalled on the cache budget (no preemption): both must agree on that too
    assert ns.num_active() == os_.num_active()
    if prefix:
        assert cached_total[0] > 0
    return steps


@pytest.mark.parametrize("policy", ["fifo", "prefill_first"])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_native_scheduler_matches_oracle(policy, seed):
    _drive(seed, policy, num_blocks=4000, bs=16, max_blocks=64, budget=512, cap=32, n_req=120)


@pytest.mark.parametrize("policy", ["fifo", "prefill_first"])
def test_native_scheduler_tight_pool(policy):
    # few blocks: chunks are cut to what fits and decodes wait for blocks
    _drive(11, policy, num_blocks=180, bs=8, max_blocks=96, budget=256, cap=16, n_req=60)


@pytest.mark.parametrize("policy", ["fifo", "prefill_first"])
def test_native_scheduler_with_forks_and_copy_on_write(policy):
    _drive(21, policy, num_blocks=3000, bs=4, max_blocks=200, budget=300, cap=24, n_req=60,
           fork_p=0.3)


@pytest.mark.parametrize("policy", ["fifo", "prefill_first"])
@pytest.mark.parametrize("num_blocks", [5000, 260])
def test_native_prefix_cache_matches_oracle(policy, num_blocks):
    # shared system prompts: cache hits, blocks kept after their requests end, and (small
    # pool) demotion of the most recently initialized cached blocks
    _drive(41 + num_blocks, policy, num_blocks=num_blocks, bs=16, max_blocks=40, budget=400,
           cap=16, n_req=80, prefix=True, fork_p=0.1)


def test_native_scheduler_small_cap_large_budget():
    _drive(31, "fifo", num_blocks=5000, bs=32, max_blocks=32, budget=4096, cap=3, n_req=40)


def test_native_allocator_example_and_errors():
    a = BlockAllocator(8, 4, 8)
    a.add_seq(1, 6)
    a.fork(1, 2)
    a.fork(1, 3)
    assert a.append(2, 1) == [(6, 5)] and a.append(3, 1) == [(6, 4)]
    assert a.table(2) == ([7, 5], 7) and a.table(3) == ([7, 4], 7)
    a.free_seq(1)
    assert a.ref_count(7) == 2 and a.ref_count(6) == 0 and a.num_free() == 5
    with pytest.raises(CbError):
        a.add_seq(2, 1)            # exists
    with pytest.raises(CbError):
        a.append(99, 1)            # unknown
    with pytest.raises(CbError):
        a.add_seq(50, 4 * 9)       # wider than the table
    with pytest.raises(CbError):
        BlockAllocator(8, 3, 8)    # block_size < 4
    assert a.ref_count(-1) == -1 and a.ref_count(8) == -1


def test_native_scheduler_rejects_bad_requests():
    s = Scheduler(BlockAllocator(100, 16, 4), 64, 4)
    s.add_request(0, 10, 5)
    with pytest.raises(CbError):
        s.add_request(0, 10, 5)    # duplicate id
    with pytest.raises(CbError):
        s.add_request(1, 60, 10)   # 69 tokens > 4 blocks x 16
    with pytest.raises(CbError):
        s.add_request(2, 0, 1)
    with pytest.raises(CbError):
        s.fork_request(0, 3, 5)    # parent not decoding yet
