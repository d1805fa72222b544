"""The scheduler / allocator oracle against what the pages fix.

Pins, by page and section:
  * "LLM learning path 3.3", section "Code" (the allocator demo and its expected output): a
    6-token prompt in 4-token blocks takes 2 blocks, the last half full; two forks that each
    write one token get private copies of that shared last block while the first block stays
    shared, with reference count 2 once the parent is freed.
  * Same page, section "Chunked prefill": a 10,000-token prompt with a ~1,500-token chunk is
    prefilled in about 7 steps; one token per running decode is added before the prefill chunk.
  * Same page, section "Code" (static vs continuous comparison): admitting new requests every
    step finishes the same work in fewer steps than static batching; here the scheduler's step
    count must equal list scheduling of the same lengths on B slots in arrival order.
  * transformers "Continuous batching architecture", section "Scheduler": FIFO order (decodes,
    then active prefills, then waiting requests), PrefillFirst completes split prefills before
    decode, the token budget and the request cap.
"""
import random

import pytest

from oracle.scheduler import (AllocatorError, BlockAllocator, Scheduler, block_hash, blocks_for,
                              fnv1a64)


def test_allocator_fork_copy_on_write_example():
    a = BlockAllocator(num_blocks=8, block_size=4, max_blocks_per_seq=8)
    a.add_seq("p", 6)
    assert len(a.tables["p"]) == 2 and a.lens["p"] == 6          # last block half full
    a.fork("p", "s1")
    a.fork("p", "s2")
    first, last = a.tables["p"]
    assert a.ref[first] == a.ref[last] == 3
    copies = a.append("s1", 1) + a.append("s2", 1)
    assert [c[0] for c in copies] == [last, last]                 # both copy the shared block
    for s in ("s1", "s2"):
        assert a.tables[s][0] == first                            # first block stays shared
        assert a.tables[s][1] != last and a.ref[a.tables[s][1]] == 1
    assert a.tables["s1"][1] != a.tables["s2"][1]
    a.free_seq("p")
    assert a.ref[first] == 2                                      # ref count 2 after the free
    assert a.ref[last] == 0 and last in a.free
    # free list: 8 - 2 (prompt) - 2 (copies) + 1 (the parent's private last block)
    assert len(a.free) == 5


def test_allocator_takes_the_last_free_block_first():
    a = BlockAllocator(num_blocks=5, block_size=4, max_blocks_per_seq=5)
    a.add_seq(0, 9)
    assert a.tables[0] == [4, 3, 2]                               # list.pop() order
    a.free_seq(0)
    a.add_seq(1, 1)
    assert a.tables[1] == [2]                                     # most recently freed first


def test_allocator_new_block_only_when_the_last_is_full():
    a = BlockAllocator(num_blocks=10, block_size=4, max_blocks_per_seq=10)
    a.add_seq(0, 3)
    assert a.append(0, 1) == [] and len(a.tables[0]) == 1         # fills block 0
    a.append(0, 1)
    assert len(a.tables[0]) == 2                                   # token 5 starts block 1
    a.fork(0, 1)
    a.append(0, 4)                                                 # shared, partly filled
    assert a.ref[a.tables[1][1]] == 1 and len(a.tables[0]) == 3


def test_allocator_exhaustion_and_table_width():
    a = BlockAllocator(num_blocks=2, block_size=4, max_blocks_per_seq=2)
    with pytest.raises(AllocatorError):
        a.add_seq(0, 9)
    a.add_seq(0, 8)
    with pytest.raises(AllocatorError):
        a.append(0, 1)


def _run(s, limit=100000):
    steps = []
    while s.num_active():
        steps.append(s.step())
        assert len(steps) < limit
    return steps


def test_ten_thousand_token_prompt_takes_seven_chunks_of_1500():
    s = Scheduler(BlockAllocator(2000, 16, 1000), max_batch_tokens=1500, max_requests_per_batch=8)
    s.add_request(0, 10000, 1)
    steps = _run(s)
    prefill = [b for b in steps if b["q_lens"]]
    assert [b["q_lens"][0] for b in prefill] == [1500] * 6 + [1000]
    assert len(prefill) == 7 == -(-10000 // 1500)


def test_fifo_one_token_per_decode_then_a_prefill_chunk():
    s = Scheduler(BlockAllocator(4000, 16, 1000), max_batch_tokens=512, max_requests_per_batch=64)
    for r in range(3):
        s.add_request(r, 5, 50)
    s.step()                                         # the three prompts
    s.add_request(9, 10000, 5)
    b = s.step()
    assert b["seq_ids"] == [0, 1, 2, 9]
    assert b["q_lens"] == [1, 1, 1, 509]
    assert b["num_decode"] == 3


def test_fifo_active_prefill_before_new_requests():
    s = Scheduler(BlockAllocator(4000, 16, 1000), max_batch_tokens=100, max_requests_per_batch=8)
    s.add_request(0, 250, 2)
    s.add_request(1, 30, 2)
    b1 = s.step()
    assert b1["seq_ids"] == [0] and b1["q_lens"] == [100]      # request 1 waits: budget spent
    b2 = s.step()
    assert b2["seq_ids"] == [0] and b2["q_lens"] == [100]
    b3 = s.step()
    assert b3["seq_ids"] == [0, 1] and b3["q_lens"] == [50, 30]


def test_prefill_first_puts_split_prefills_before_decodes():
    s = Scheduler(BlockAllocator(4000, 16, 1000), max_batch_tokens=64,
                  max_requests_per_batch=8, policy="prefill_first")
    s.add_request(0, 4, 10)
    s.step()                                          # request 0 now decodes
    s.add_request(1, 200, 2)
    s.step()                                          # request 1 starts: 0 decodes, 1 prefills
    # the split prefill takes the whole budget until it completes; decode resumes after it
    assert [(b["seq_ids"], b["q_lens"]) for b in (s.step(), s.step(), s.step())] == [
        ([1], [64]), ([1], [64]), ([1, 0], [9, 1])]
    f = Scheduler(BlockAllocator(4000, 16, 1000), max_batch_tokens=64, max_requests_per_batch=8)
    f.add_request(0, 4, 10)
    f.step()
    f.add_request(1, 200, 2)
    f.step()
    b = f.step()
    assert b["seq_ids"] == [0, 1] and b["q_lens"] == [1, 63]


def test_request_cap_and_token_budget_hold():
    rng = random.Random(5)
    s = Scheduler(BlockAllocator(600, 8, 200), max_batch_tokens=97, max_requests_per_batch=7)
    for r in range(40):
        s.add_request(r, rng.randint(1, 300), rng.randint(1, 40))
    for b in _run(s):
        assert len(b["seq_ids"]) <= 7 and sum(b["q_lens"]) <= 97


def test_every_request_feeds_prompt_plus_new_minus_one_tokens():
    rng = random.Random(6)
    s = Scheduler(BlockAllocator(300, 4, 400), max_batch_tokens=64, max_requests_per_batch=5)
    want = {}
    for r in range(30):
        p, n = rng.randint(1, 100), rng.randint(1, 30)
        s.add_request(r, p, n)
        want[r] = p + n - 1
    fed = {r: 0 for r in want}
    last_kv = {}
    for b in _run(s):
        for sid, q, kv in zip(b["seq_ids"], b["q_lens"], b["kv_lens"]):
            fed[sid] += q
            assert kv == last_kv.get(sid, 0) + q          # kv_len counts this step's tokens
            last_kv[sid] = kv
    assert fed == want
    assert len(s.alloc.free) == 300 and not s.alloc.tables


def test_decode_waits_when_no_block_is_free():
    s = Scheduler(BlockAllocator(2, 4, 4), max_batch_tokens=16, max_requests_per_batch=4)
    s.add_request(0, 4, 3)
    s.add_request(1, 4, 3)
    b = s.step()
    assert b["q_lens"] == [4, 4]                      # both prompts fill one block each
    b = s.step()
    assert b["seq_ids"] == []                         # each decode needs a new block: none free


def test_continuous_is_list_scheduling_and_beats_static():
    # a stream like the page's comparison: 256 requests, exponential lengths of mean ~200
    # capped at 2000, 16 slots
    import numpy as np
    lens = [int(x) for x in np.minimum(np.random.default_rng(0).exponential(200, 256) + 1, 2000)]
    B = 16
    static = sum(max(lens[i:i + B]) for i in range(0, len(lens), B))
    # continuous batching as the page describes it: B slots, a finished request's slot is
    # refilled by the next waiting request at the next step; a request of length L holds its
    # slot for L steps.  That is list scheduling in arrival order on B slots.
    import heapq
    free_at = [0] * B
    cont = 0
    for L in lens:
        t = heapq.heappop(free_at)
        heapq.heappush(free_at, t + L)
        cont = max(cont, t + L)
    # the scheduler with one-token prompts: a request of L new tokens is in L steps
    s = Scheduler(BlockAllocator(100000, 16, 200), max_batch_tokens=4096, max_requests_per_batch=B)
    for i, L in enumerate(lens):
        s.add_request(i, 1, L)
    steps = [b for b in _run(s)]
    busy = [b for b in steps if b["seq_ids"]]
    assert len(busy) == cont
    assert cont < static
    assert sum(lens) / (B * cont) > sum(lens) / (B * static)


def test_blocks_for_matches_the_printed_examples():
    assert blocks_for(1000, 16) == 63 and blocks_for(8192, 256) == 32


# ------------------------------------------------------------------------------ prefix caching

def test_fnv1a64_published_vectors():
    # the FNV authors' test vectors for 64-bit FNV-1a
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_chains_the_prefix():
    a, b = [1, 2, 3, 4], [5, 6, 7, 8]
    assert block_hash(0, a) != block_hash(0, b)
    assert block_hash(block_hash(0, a), b) != block_hash(block_hash(0, b), b)  # same block, other prefix
    assert block_hash(7, a) == fnv1a64((7).to_bytes(8, "little") + bytes([1, 0, 0, 0, 2, 0, 0, 0,
                                                                         3, 0, 0, 0, 4, 0, 0, 0]))


def _prefix_sched(num_blocks=400, bs=16, budget=4096, cap=8):
    return Scheduler(BlockAllocator(num_blocks, bs, 200, prefix_caching=True), budget, cap)


def test_shared_system_prompt_skips_its_prefill():
    # the page's example: a 1,000-token system prompt S shared by three requests; the first
    # misses, the later ones skip ~1,000 tokens of prefill (whole blocks of S here)
    rng = random.Random(3)
    S = [rng.randrange(50000) for _ in range(1000)]
    r1 = S + [11, 12, 13, 14]
    r2 = S + [11, 12, 15]
    r3 = S + [rng.randrange(50000) for _ in range(200)]
    s = _prefix_sched()
    s.add_request(1, len(r1), 2, r1)
    b = s.step()
    assert b["q_lens"] == [1004] and b["cached"] == 0
    s.add_request(2, len(r2), 2, r2)
    s.add_request(3, len(r3), 2, r3)
    b = s.step()
    prefill = dict(zip(b["seq_ids"], b["q_lens"]))
    assert b["cached"] == 2 * 992                      # 62 full blocks of S each
    assert prefill[2] == len(r2) - 992 and prefill[3] == len(r3) - 992
    t1 = s.alloc.tables[1]
    assert s.alloc.tables[2][:62] == t1[:62] == s.alloc.tables[3][:62]
    assert all(s.alloc.ref[x] == 3 for x in t1[:62])


def test_a_match_leaves_the_last_token_to_compute():
    toks = list(range(64))                             # exactly 4 blocks of 16
    s = _prefix_sched()
    s.add_request(1, 64, 1, toks)
    s.step()
    s.add_request(2, 64, 1, toks)
    b = s.step()
    assert b["seq_ids"] == [2] and b["q_lens"] == [16] and b["cached"] == 48


def test_cached_blocks_outlive_their_requests_and_are_reused():
    toks = list(range(100, 164))
    s = _prefix_sched()
    s.add_request(1, 64, 1, toks)
    s.step()
    s.step()                                           # retires request 1
    assert not s.alloc.tables and s.alloc.num_free() == 400
    assert len(s.alloc.idle) == 4                      # its 4 prompt blocks keep their content
    s.add_request(2, 64 + 5, 1, toks + [1, 2, 3, 4, 5])
    b = s.step()
    assert b["cached"] == 64 and b["q_lens"] == [5]


def test_eviction_demotes_the_most_recently_initialized_block_first():
    s = _prefix_sched(num_blocks=6, bs=4, cap=4)
    a_toks, b_toks = [1] * 8 + [9], [2] * 8 + [9]      # 2 cacheable blocks + 1 partial each
    s.add_request(1, 9, 1, a_toks)
    s.step()
    s.add_request(2, 9, 1, b_toks)
    s.step()                                           # retires 1, prefills 2
    s.step()                                           # retires 2
    al = s.alloc
    order = sorted(al.idle, key=lambda x: al.born[x])
    assert len(order) == 4 and al.num_free() == 6
    # 2 blocks without content left; a 16-token sequence needs 4: the two most recently
    # initialized cached blocks (request 2's) are demoted first
    al.add_seq(99, 16)
    assert set(al.tables[99]) >= set(order[2:])
    assert set(order[:2]) <= al.idle                   # request 1's prefix is still cached
    al.free_seq(99)
    s.add_request(3, 9, 1, a_toks)
    assert s.step()["cached"] == 8
