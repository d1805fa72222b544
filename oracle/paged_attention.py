"""Oracle: paged KV-append and ragged paged attention, float64 numpy.

TEST INFRASTRUCTURE (see the package docstring): nothing in the CUDA library
uses this file.

Sources, by page title and section:
  * "LLM learning path 3.3 Batching & Memory Management", section
    "PagedAttention: block tables": entry j of a sequence's block table is the
    physical block holding tokens [j*bs, (j+1)*bs); token position p lives in
    block table[p // bs] at offset p % bs (worked example: table [7, 2, 5],
    bs 4, token 9 -> block 5, offset 1).  The page text lost the formula in
    extraction; the worked example fixes it.
  * "Continuous batching in transformers", section "The paged cache, its two
    reserved blocks, and the block-size trade": a page is the K (or V) state
    of one token in one layer, a block is block_size pages, and the physical
    tensor is token-major [(blocks) * block_size, kv_heads, head_dim].  The
    reserved padding blocks serve padded CUDA-graph tokens, which a ragged
    batch does not have, so they are not modelled; block_size < 4 is rejected.
  * "LLM learning path 3.3", section "Continuous (iteration-level) batching"
    and "Continuous batching from first principles" (summary): all tokens of
    a step are packed into one ragged axis with per-sequence lengths, and
    attention is restricted to each token's own sequence.
  * "LLM learning path 3.3", section "Chunked prefill": a chunk of queries
    attends to a cache that already holds the earlier chunks, so query i of a
    chunk whose prior context is ctx sees keys 0 .. ctx + i (the causal mask
    offset by the prior context).
  * Continuous-batching architecture doc, section "Memory management": each
    request holds the block ids the attention kernel reads from and writes to;
    here the write (append) happens before the read (attention).

Readings where the pages are silent (each also listed in the design notes):
  * GQA: query head h reads KV head h // (Hq / Hkv).
  * kv_lens count the keys visible after this step's append, so the prior
    context of sequence s is kv_lens[s] - q_len[s].
  * A sequence with q_len == 0 contributes nothing; kv_len < q_len is an error.
"""
from __future__ import annotations

import numpy as np

MIN_BLOCK_SIZE = 4


class OracleError(ValueError):
    """Raised for metadata the method does not define (bad slots, lengths, sizes)."""


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bf16 bit patterns (a bf16 is the top half of a float32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_block_size(block_size: int) -> int:
    bs = int(block_size)
    if bs < MIN_BLOCK_SIZE:
        raise OracleError(f"block_size must be >= {MIN_BLOCK_SIZE}, got {bs}")
    return bs


def slot_of(table_row, pos: int, block_size: int, num_pages: int | None = None) -> int:
    """Flat token slot of position ``pos``: physical block table[pos // bs], offset pos % bs."""
    bs = _check_block_size(block_size)
    if pos < 0:
        raise OracleError(f"negative position {pos}")
    logical_block, offset = divmod(int(pos), bs)
    if logical_block >= len(table_row):
        raise OracleError(f"position {pos} needs logical block {logical_block}, table has {len(table_row)}")
    physical = int(table_row[logical_block])
    if physical < 0 or (num_pages is not None and physical >= num_pages):
        raise OracleError(f"block id {physical} outside the pool")
    return physical * bs + offset


def _seq_bounds(cu_seqlens_q, kv_lens):
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    kv = np.asarray(kv_lens, dtype=np.int64)
    if cu.ndim != 1 or kv.ndim != 1 or cu.shape[0] != kv.shape[0] + 1:
        raise OracleError("cu_seqlens_q must have one more entry than kv_lens")
    if cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise OracleError("cu_seqlens_q must start at 0 and be non-decreasing")
    q_len = np.diff(cu)
    if np.any(kv < q_len):
        raise OracleError("kv_len < q_len: the appended tokens must be part of the visible keys")
    return cu, kv, q_len


def kv_append(k_new, v_new, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size):
    """Scatter this step's K/V rows into their pages; returns new (k_pages, v_pages) bit arrays.

    Token i of sequence s (packed index cu[s] + i) sits at absolute position
    ctx_s + i with ctx_s = kv_len_s - q_len_s, and lands in slot_of(table[s], pos).
    The copy is of bf16 bit patterns, so it is exact.  Raises before writing
    anything if any destination is undefined or two tokens share a slot, or if
    a token would write into a block that another sequence maps within its
    visible keys (a write to a shared block needs copy-on-write first, which is
    the block manager's job, not this pass's).
    """
    bs = _check_block_size(block_size)
    cu, kv, q_len = _seq_bounds(cu_seqlens_q, kv_lens)
    kp = np.array(k_pages, dtype=np.uint16, copy=True)
    vp = np.array(v_pages, dtype=np.uint16, copy=True)
    P = kp.shape[0]
    if kp.shape[1] != bs or vp.shape != kp.shape:
        raise OracleError("page tensors must be [P, block_size, Hkv, D] and alike")
    table = np.asarray(block_table)
    S = kv.shape[0]
    if np.asarray(k_new).shape[0] != cu[-1]:
        raise OracleError("k_new must have cu_seqlens_q[-1] rows")

    # Blocks each sequence can read: the first ceil(kv_len / bs) table entries.
    readers: dict[int, set[int]] = {}
    for s in range(S):
        for j in range(-(-int(kv[s]) // bs)):
            readers.setdefault(int(table[s, j]), set()).add(s)

    dest = {}
    for s in range(S):
        ctx = int(kv[s] - q_len[s])
        for i in range(int(q_len[s])):
            slot = slot_of(table[s], ctx + i, bs, P)
            if slot in dest:
                raise OracleError(f"slot {slot} written twice")
            block = slot // bs
            if readers.get(block, {s}) - {s}:
                raise OracleError(f"token of sequence {s} would write shared block {block}")
            dest[slot] = int(cu[s]) + i

    flat_k = kp.reshape(P * bs, *kp.shape[2:])
    flat_v = vp.reshape(P * bs, *vp.shape[2:])
    for slot, t in dest.items():
        flat_k[slot] = k_new[t]
        flat_v[slot] = v_new[t]
    return kp, vp


def gather_kv(pages, table_row, kv_len: int, block_size: int) -> np.ndarray:
    """float64 [kv_len, Hkv, D]: row j is the page at slot_of(table_row, j)."""
    bs = _check_block_size(block_size)
    P = pages.shape[0]
    flat = np.asarray(pages).reshape(P * bs, *pages.shape[2:])
    n = int(kv_len)
    if n == 0:
        return np.zeros((0,) + pages.shape[2:], dtype=np.float64)
    row = np.asarray(table_row, dtype=np.int64)
    j = np.arange(n)
    logical = j // bs
    if logical[-1] >= row.shape[0]:
        raise OracleError(f"kv_len {n} needs {logical[-1] + 1} blocks, table has {row.shape[0]}")
    physical = row[logical]
    if physical.min() < 0 or physical.max() >= P:
        raise OracleError("block id outside the pool")
    slots = physical * bs + j % bs   # the same rule as slot_of, for every key at once
    return bf16_bits_to_f64(flat[slots])


def stable_softmax(x: np.ndarray, axis: int = -1):
    """(softmax(x), natural log-sum-exp of x) along ``axis``, with the max subtracted first."""
    m = np.max(x, axis=axis, keepdims=True)
    e = np.exp(x - m)
    z = np.sum(e, axis=axis, keepdims=True)
    return e / z, np.squeeze(m + np.log(z), axis=axis)


def attention_one_sequence(q, K, V, ctx: int, scale: float, window: int = 0):
    """Exact causal attention of one sequence's queries over its gathered keys.

    q [n, Hq, D] float64 (query i at absolute position ctx + i),
    K, V [kv, Hkv, D] float64 with kv >= ctx + n.
    window > 0: sliding window, query at position p sees keys j with p - window < j <= p.
    Returns out [n, Hq, D] and lse [n, Hq] (natural log of the softmax normaliser
    of the scaled scores).
    """
    n, Hq, D = q.shape
    kv, Hkv, _ = K.shape
    if Hq % Hkv:
        raise OracleError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    out = np.zeros((n, Hq, D), dtype=np.float64)
    lse = np.zeros((n, Hq), dtype=np.float64)
    if n == 0:
        return out, lse
    # visible[i, j]: key j is at or before query i's absolute position ctx + i.
    pos = (ctx + np.arange(n))[:, None]
    visible = np.arange(kv)[None, :] <= pos
    if window > 0:
        visible &= np.arange(kv)[None, :] > pos - window
    for h in range(Hq):
        g = h // G
        scores = scale * (q[:, h, :] @ K[:, g, :].T)            # [n, kv]
        scores = np.where(visible, scores, -np.inf)
        p, lse[:, h] = stable_softmax(scores, axis=1)
        out[:, h, :] = p @ V[:, g, :]
    return out, lse


def ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                           block_size: int, scale: float, window: int = 0):
    """Attention over a ragged batch whose K/V live in pages.

    q: bf16 bits [T, Hq, D]; pages: bf16 bits [P, bs, Hkv, D] (after the append).
    Returns float64 out [T, Hq, D] and lse [T, Hq].
    """
    bs = _check_block_size(block_size)
    cu, kv, q_len = _seq_bounds(cu_seqlens_q, kv_lens)
    q = np.asarray(q)
    T, Hq, D = q.shape
    if cu[-1] != T:
        raise OracleError("cu_seqlens_q[-1] must equal the number of query rows")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.zeros((T, Hq), dtype=np.float64)
    for s in range(kv.shape[0]):
        n = int(q_len[s])
        if n == 0:
            continue
        K = gather_kv(k_pages, block_table[s], int(kv[s]), bs)
        V = gather_kv(v_pages, block_table[s], int(kv[s]), bs)
        qs = bf16_bits_to_f64(q[cu[s]:cu[s] + n])
        o, l = attention_one_sequence(qs, K, V, int(kv[s]) - n, scale, window)
        out[cu[s]:cu[s] + n] = o
        lse[cu[s]:cu[s] + n] = l
    return out, lse


def attention_rows(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size: int,
                   scale: float, rows, window: int = 0):
    """out/lse for selected (token, head) pairs only: [(t, h), ...] -> (out [n, D], lse [n]).

    Used to check a sample of a batch too large to run whole; each row is the
    same definition as ``ragged_paged_attention``.
    """
    bs = _check_block_size(block_size)
    cu, kv, q_len = _seq_bounds(cu_seqlens_q, kv_lens)
    Hq = q.shape[1]
    Hkv = k_pages.shape[2]
    G = Hq // Hkv
    res_o, res_l = [], []
    cache = {}
    for t, h in rows:
        s = int(np.searchsorted(cu, t, side="right") - 1)
        i = t - int(cu[s])
        ctx = int(kv[s] - q_len[s])
        if s not in cache:
            cache = {s: (gather_kv(k_pages, block_table[s], int(kv[s]), bs),
                         gather_kv(v_pages, block_table[s], int(kv[s]), bs))}
        K, V = cache[s]
        g = h // G
        qv = bf16_bits_to_f64(q[t, h])
        lo = max(0, ctx + i + 1 - window) if window > 0 else 0
        x = scale * (K[lo: ctx + i + 1, g, :] @ qv)
        p, l = stable_softmax(x)
        res_o.append(p @ V[lo: ctx + i + 1, g, :])
        res_l.append(float(l))
    return np.asarray(res_o), np.asarray(res_l)
