"""Oracle: the batching arithmetic the pages print, as plain integer functions.

TEST INFRASTRUCTURE (see the package docstring).

Sources, by page title and section:
  * "Continuous batching in transformers", section "Why use it": a padded
    batch is a rectangle (rows x longest row); packing the same rows raggedly
    stores only the real tokens; one n-token prompt joining B-1 one-token
    decodes wastes (n-1)(B-1) slots, which is bilinear, not quadratic; a
    zero-length row is not a batch and must be rejected.
  * "LLM learning path 3.3 Batching & Memory Management", section "Static
    batching and its waste": static-batch utilisation is the useful
    token-steps over B * max_i N_i (the page's formula was lost in extraction;
    its worked numbers 670/2000 and 1300/4000 fix it).
  * "Continuous batching in transformers", section "The paged cache, its two
    reserved blocks, and the block-size trade", and "LLM learning path 3.3",
    section "Check your understanding": a sequence of L tokens occupies
    ceil(L / bs) blocks and wastes the unused tail of its last block.
"""
from __future__ import annotations

from .paged_attention import MIN_BLOCK_SIZE, OracleError


def _rows(lengths) -> list[int]:
    rows = [int(x) for x in lengths]
    if not rows:
        raise OracleError("a batch needs at least one row")
    if min(rows) <= 0:
        raise OracleError("every row of a batch needs at least one token")
    return rows


def padded_slots(lengths) -> int:
    """Token slots of the rectangular (padded) batch: number of rows times the longest row."""
    rows = _rows(lengths)
    return len(rows) * max(rows)


def useful_slots(lengths) -> int:
    """Token slots of the ragged (packed) batch: exactly the real tokens."""
    return sum(_rows(lengths))


def padding_waste(B: int, n: int) -> int:
    """Pad slots when one n-token prompt is batched with B-1 single-token decodes."""
    if B < 1 or n < 1:
        raise OracleError("need B >= 1 and n >= 1")
    lengths = [n] + [1] * (B - 1)
    return padded_slots(lengths) - useful_slots(lengths)


def static_utilisation(output_lengths) -> float:
    """Useful token-steps over slot-steps of a static batch that runs until its longest row ends."""
    return useful_slots(output_lengths) / padded_slots(output_lengths)


def blocks_for(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of num_tokens occupies: the ceiling of num_tokens / block_size."""
    if block_size < MIN_BLOCK_SIZE:
        raise OracleError(f"block_size must be >= {MIN_BLOCK_SIZE}")
    if num_tokens < 0:
        raise OracleError("negative token count")
    full, rest = divmod(int(num_tokens), int(block_size))
    return full + (1 if rest else 0)


def tail_waste(num_tokens: int, block_size: int) -> int:
    """Slots paid for but unused: the empty tail of the last block."""
    return blocks_for(num_tokens, block_size) * int(block_size) - int(num_tokens)
