"""CPU oracle for ragged paged attention and the paged KV-append.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
smoke check and the CPU-baseline leg of the benchmark may import this package.
The CUDA library never links, loads or calls it, and it shares no code with
the CUDA path: inputs come from the seeded generators in ``workloads``.

Everything is plain numpy in float64: the plain definition of exact attention,
written out per sequence and per head over K/V gathered through the block
table, plus the small batching arithmetic the pages print.

Pins (what each function is checked against, in tests/test_oracle_*.py):
  * ``slot_of`` / ``kv_append``: the worked block-table example of
    "LLM learning path 3.3", section "PagedAttention: block tables"
    (table [7, 2, 5], block size 4, token 9 -> block 5, offset 1), plus a
    brute-force inverse map over every written slot.
  * ``ragged_paged_attention``: textbook causal softmax attention from
    torch.nn.functional.scaled_dot_product_attention in float64 on a single
    contiguous sequence; closed forms (kv_len 1 -> v0; q = 0 -> mean of the
    visible V rows; identical keys -> mean of V); explicit Python-float loops
    on tiny inputs; the invariants ragged == each sequence alone, page
    permutation, shared prefix == duplicated copy, convex-hull bound, and
    softmax shift invariance.
  * ``batching``: the values "Continuous batching in transformers" and
    "LLM learning path 3.3" print (693 wasted slots, 670/2000, 1300/4000,
    63 blocks with 8 wasted slots, 32 x 256 = 8192, ...).
  * ``scheduler``: the allocator demo of "LLM learning path 3.3", section "Code" (forked
    samples copy the shared last block, the first block keeps count 2 after the parent is
    freed), the 10,000-token / 1,500-token chunking example, the FIFO and PrefillFirst orders
    of the transformers "Scheduler" section, and continuous batching = list scheduling on B
    slots, fewer steps than static batching (tests/test_oracle_scheduler.py).
  * ``blocks``: element-wise brute force on tiny pools (tests/test_oracle_blocks.py).
No function here is "parity unpinned".
"""
from .paged_attention import (  # noqa: F401
    OracleError,
    bf16_bits_to_f64,
    slot_of,
    kv_append,
    gather_kv,
    stable_softmax,
    attention_one_sequence,
    ragged_paged_attention,
    attention_rows,
)
from . import batching  # noqa: F401
from . import blocks  # noqa: F401
from . import scheduler  # noqa: F401
