"""Seeded synthetic batches for the ragged paged-attention path.

This module only draws inputs: random bf16 values, sequence lengths, a shuffled
page pool and block tables.  It holds none of the method's arithmetic (no slot
mapping, no attention); both the CUDA path and the oracle consume what it
produces, and neither is imported here.

Layouts (all C-contiguous, bf16 values carried as uint16 bit patterns):

  q, out         [T, Hq, D]        T = cu_seqlens_q[S], the packed (ragged) token axis
  k_new, v_new   [T, Hkv, D]       the K/V of this step's tokens, appended before attention
  k_pages,v_pages[P, bs, Hkv, D]   token-major pages: page = one token's K (or V),
                                   block = bs consecutive pages ("Continuous batching in
                                   transformers", section "The paged cache, its two reserved
                                   blocks, and the block-size trade")
  block_table    [S, max_blocks]   int32, entry j = physical block of tokens [j*bs, (j+1)*bs);
                                   unused entries are -1
  cu_seqlens_q   [S+1]             int32 prefix of per-sequence query counts
  kv_lens        [S]               int32 keys visible to the sequence AFTER this step's append

Poison: every slot that is not part of a sequence's prior context holds a bf16
NaN (unreferenced pages, slots at or beyond kv_len, and the slots this step's
append is about to fill), so a stray read or a missing append shows up as NaN.

The five named workloads mirror the batches the pages talk about (decode
tokens and chunked-prefill chunks packed into one token axis, block sizes 16 to
64, GQA with 8 KV heads at head_dim 128); their parameters are listed in
``CONFIGS``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bit patterns.

    For finite inputs u + 0x7FFF + 1 stays below 2^32, so uint32 arithmetic is exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_x = x.reshape(-1).view(np.uint32)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_x.size, step):
        u = flat_x[i:i + step].copy()
        lsb = (u >> 16) & 1
        u += 0x7FFF
        u += lsb
        u >>= 16
        flat_o[i:i + step] = u
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


@dataclasses.dataclass
class Batch:
    name: str
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    k_pages: np.ndarray
    v_pages: np.ndarray
    block_table: np.ndarray
    cu_seqlens_q: np.ndarray
    kv_lens: np.ndarray
    block_size: int
    scale: float
    num_q_heads: int
    num_kv_heads: int
    head_dim: int

    @property
    def num_seqs(self) -> int:
        return int(self.kv_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)


def _draw(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values rounded to bf16, drawn in row-major order in chunks of 2^24."""
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat.size, step):
        n = min(step, flat.size - i)
        x = rng.standard_normal(size=n, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        flat[i:i + n] = f32_to_bf16_bits(x)
    return out


@dataclasses.dataclass
class Layout:
    """The metadata of a batch without its values: lengths, block tables and shapes."""
    name: str
    block_table: np.ndarray
    cu_seqlens_q: np.ndarray
    kv_lens: np.ndarray
    block_size: int
    scale: float
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_pages: int
    k_scale: float

    @property
    def num_seqs(self) -> int:
        return int(self.kv_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)


def _layout(rng, q_lens, kv_lens, num_q_heads, num_kv_heads, head_dim, block_size, *,
            num_pages=None, pool_factor=1.25, k_scale=1.0, shared_prefix=None, slack_blocks=2,
            max_blocks=None, scale=None, shuffle_pages=True, name="custom"):
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    S = len(q_lens)
    assert kv_lens.shape == (S,)
    assert np.all(q_lens >= 0) and np.all(kv_lens >= q_lens)
    bs = int(block_size)
    nblk = (kv_lens + bs - 1) // bs
    shared_members: set[int] = set()
    n_shared_blocks = 0
    if shared_prefix is not None:
        members, n_tok = shared_prefix
        assert n_tok % bs == 0
        n_shared_blocks = n_tok // bs
        shared_members = set(int(m) for m in members)
        for m in shared_members:
            assert kv_lens[m] - q_lens[m] >= n_tok
    needed = int(nblk.sum()) - (max(len(shared_members) - 1, 0) * n_shared_blocks)
    if num_pages is None:
        num_pages = max(int(math.ceil(pool_factor * needed)), 1)
    assert num_pages >= needed, (num_pages, needed)
    if max_blocks is None:
        max_blocks = int(nblk.max(initial=0)) + slack_blocks
    max_blocks = max(int(max_blocks), 1)
    assert max_blocks >= int(nblk.max(initial=0))

    page_ids = rng.permutation(num_pages) if shuffle_pages else np.arange(num_pages)
    table = np.full((S, max_blocks), -1, dtype=np.int32)
    nxt = 0
    shared_ids = None
    if n_shared_blocks:
        shared_ids = page_ids[:n_shared_blocks].astype(np.int32)
        nxt = n_shared_blocks
    for s in range(S):
        start = 0
        if s in shared_members:
            table[s, :n_shared_blocks] = shared_ids
            start = n_shared_blocks
        cnt = int(nblk[s]) - start
        table[s, start:start + cnt] = page_ids[nxt:nxt + cnt]
        nxt += cnt

    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(int(head_dim))
    return Layout(name=name, block_table=table, cu_seqlens_q=cu,
                  kv_lens=kv_lens.astype(np.int32), block_size=bs, scale=float(scale),
                  num_q_heads=int(num_q_heads), num_kv_heads=int(num_kv_heads),
                  head_dim=int(head_dim), num_pages=int(num_pages), k_scale=float(k_scale))


def batch_layout(q_lens, kv_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, seed: int, **kw) -> Layout:
    """The metadata build_batch would draw with the same arguments (the same block tables),
    without drawing any values: for callers that fill the values elsewhere."""
    return _layout(np.random.default_rng(seed), q_lens, kv_lens, num_q_heads, num_kv_heads,
                   head_dim, block_size, **kw)


def build_batch(
    q_lens,
    kv_lens,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int,
    seed: int,
    *,
    num_pages: int | None = None,
    pool_factor: float = 1.25,
    k_scale: float = 1.0,
    shared_prefix: tuple[list[int], int] | None = None,
    slack_blocks: int = 2,
    max_blocks: int | None = None,
    scale: float | None = None,
    shuffle_pages: bool = True,
    name: str = "custom",
) -> Batch:
    """Draw one ragged batch.

    q_lens[s] query tokens of sequence s are appended this step, so its prior
    context is kv_lens[s] - q_lens[s] tokens, already in the cache.
    ``shared_prefix=(members, n_tokens)`` makes the listed sequences point at the
    same physical blocks for their first n_tokens (n_tokens must be a whole
    number of blocks and every member must have at least that much prior context).
    """
    rng = np.random.default_rng(seed)
    lay = _layout(rng, q_lens, kv_lens, num_q_heads, num_kv_heads, head_dim, block_size,
                  num_pages=num_pages, pool_factor=pool_factor, k_scale=k_scale,
                  shared_prefix=shared_prefix, slack_blocks=slack_blocks, max_blocks=max_blocks,
                  scale=scale, shuffle_pages=shuffle_pages, name=name)
    table, cu, bs, num_pages = lay.block_table, lay.cu_seqlens_q, lay.block_size, lay.num_pages
    kv_lens = lay.kv_lens.astype(np.int64)
    q_lens = np.diff(cu).astype(np.int64)
    S = lay.num_seqs
    nblk = (kv_lens + bs - 1) // bs
    H, Hkv, D = lay.num_q_heads, lay.num_kv_heads, lay.head_dim
    T = int(q_lens.sum())

    # Referenced pages receive random content; everything else is poison.
    referenced = np.unique(table[table >= 0])
    k_pages = np.full((num_pages, bs, Hkv, D), BF16_NAN, dtype=np.uint16)
    v_pages = np.full((num_pages, bs, Hkv, D), BF16_NAN, dtype=np.uint16)
    if referenced.size:
        k_pages[referenced] = _draw(rng, (referenced.size, bs, Hkv, D), k_scale)
        v_pages[referenced] = _draw(rng, (referenced.size, bs, Hkv, D))
    # (referenced pages are drawn in ascending page-id order, K first, then V)
    # Poison every slot outside each sequence's prior context [0, ctx).  Shared
    # blocks are full prior context for all members, so this never touches them.
    for s in range(S):
        ctx = int(kv_lens[s] - q_lens[s])
        for blk_idx in range(int(nblk[s])):
            lo = blk_idx * bs
            first_bad = max(ctx - lo, 0)
            if first_bad < bs:
                pid = table[s, blk_idx]
                k_pages[pid, first_bad:] = BF16_NAN
                v_pages[pid, first_bad:] = BF16_NAN

    q = _draw(rng, (T, H, D))
    k_new = _draw(rng, (T, Hkv, D), k_scale)
    v_new = _draw(rng, (T, Hkv, D))
    return Batch(name=name, q=q, k_new=k_new, v_new=v_new, k_pages=k_pages, v_pages=v_pages,
                 block_table=table, cu_seqlens_q=cu, kv_lens=kv_lens.astype(np.int32),
                 block_size=bs, scale=lay.scale, num_q_heads=H, num_kv_heads=Hkv, head_dim=D)


# Named workloads.  "ctx" is the prior context, so kv_len = ctx + q_len.
CONFIGS = {
    1: "tiny ragged: 1 chunk of 32 at ctx 0 + decodes at ctx 17/64/100; 4q/2kv heads, D64, bs16, 24 shuffled pages",
    2: "decode-only: 64 seqs x 1 token, kv ~ U[512,4096]; 32q/8kv heads, D128, bs32, 16384-page pool",
    3: "mixed at 2048 tokens: 120 decodes (ctx ~ U[256,8192]) + one 1928-token chunk at ctx 3000; 32q/8kv, D128, bs32",
    4: "chunked-prefill-heavy: 16 decodes + 8 chunks of 512 (ctx ~ U[0,8192]); 32q/8kv, D128, bs64, K x4",
    5: "long-tail decode + prefix sharing: 256 seqs, kv lognormal(median 2048, sigma 1, cap 32768), 64q/8kv, D128, bs64, seqs 0-63 share 1024 tokens",
}


def config_lengths(n: int, seed: int):
    """(q_lens, kv_lens, extra kwargs for build_batch) of named workload ``n``."""
    rng = np.random.default_rng(seed + 7919)
    if n == 1:
        q = [32, 1, 1, 1]
        kv = [32, 18, 65, 101]
        return q, kv, dict(num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                           num_pages=24, scale=1.0 / 8.0)
    if n == 2:
        kv = rng.integers(512, 4096, size=64, endpoint=True)
        return [1] * 64, kv, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                                  num_pages=16384)
    if n == 3:
        ctx = rng.integers(256, 8192, size=120, endpoint=True)
        q = [1] * 120 + [1928]
        kv = list(ctx + 1) + [3000 + 1928]
        return q, kv, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32)
    if n == 4:
        dctx = rng.integers(0, 8192, size=16, endpoint=True)
        cctx = rng.integers(0, 8192, size=8, endpoint=True)
        q = [1] * 16 + [512] * 8
        kv = list(dctx + 1) + list(cctx + 512)
        return q, kv, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=64,
                           k_scale=4.0)
    if n == 5:
        z = rng.standard_normal(256)
        kv = np.clip(np.rint(2048.0 * np.exp(z)), 1, 32768).astype(np.int64)
        kv[:64] = np.maximum(kv[:64], 1025)  # sharers keep the shared 1024 tokens as prior context
        return [1] * 256, kv, dict(num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=64,
                                   shared_prefix=(list(range(64)), 1024))
    raise ValueError(f"unknown workload {n}")


def make_config(n: int, seed: int | None = None) -> Batch:
    """Named workload ``n`` (1..5) drawn with ``seed`` (default 1000 + n)."""
    if seed is None:
        seed = 1000 + n
    q, kv, kw = config_lengths(n, seed)
    return build_batch(q, kv, seed=seed, name=f"config{n}", **kw)


def make_layout(n: int, seed: int | None = None, **overrides) -> Layout:
    """The metadata of named workload ``n`` (the block tables make_config draws with the same
    seed), with optional shape overrides (head counts, head_dim, block_size)."""
    if seed is None:
        seed = 1000 + n
    q, kv, kw = config_lengths(n, seed)
    kw.update(overrides)
    return batch_layout(q, kv, seed=seed, name=f"config{n}", **kw)
