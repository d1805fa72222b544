"""Oracle: whole-block moves of the paged KV cache, as plain numpy copies of bit patterns.

TEST INFRASTRUCTURE (see the package docstring).

Sources, by page title and section:
  * "LLM learning path 3.3 Batching & Memory Management", section "PagedAttention: block
    tables": before a sequence writes into a block whose reference count is above 1, the
    engine copies that block and points the sequence's table at the copy (copy-on-write);
    section "Code": the real engine copies the KV data too.  copy_blocks is that data copy.
  * transformers "Continuous batching architecture", section "Memory management": an
    offloaded request's blocks move to CPU memory in one batched copy and back.  gather_blocks
    and scatter_blocks are that move, with the host side laid out block after block.

Pools are uint16 arrays [P, bs, Hkv, D] of bf16 bit patterns (one per K and V).
"""
from __future__ import annotations

import numpy as np


def copy_blocks(pool: np.ndarray, src, dst) -> np.ndarray:
    """A copy of `pool` in which block dst[i] holds what block src[i] held before any copy."""
    src, dst = [int(x) for x in src], [int(x) for x in dst]
    if set(src) & (set(dst) - {s for s, d in zip(src, dst) if s == d}):
        raise ValueError("a block is both read and written")
    out = pool.copy()
    for s, d in zip(src, dst):
        out[d] = pool[s]
    return out


def gather_blocks(pool: np.ndarray, blocks) -> np.ndarray:
    """Blocks listed in `blocks`, in list order: [n, bs, Hkv, D]."""
    return np.stack([pool[int(b)] for b in blocks]) if len(blocks) else pool[:0].copy()


def scatter_blocks(pool: np.ndarray, blocks, host: np.ndarray) -> np.ndarray:
    """A copy of `pool` with block blocks[i] replaced by host[i]."""
    out = pool.copy()
    for i, b in enumerate(blocks):
        out[int(b)] = host[i]
    return out
