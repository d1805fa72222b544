"""Oracle: the paged-KV block allocator and the continuous-batching schedulers, in plain Python.

TEST INFRASTRUCTURE (see the package docstring).

Sources, by page title and section:
  * "LLM learning path 3.3 Batching & Memory Management", section "Code": the allocator keeps
    a list of free block ids and takes the last one (so a fresh pool hands out the highest id
    first and a freed block is the next one reused), a reference count per block, and a block
    table and a token count per sequence.  A new sequence of n tokens takes ceil(n / bs)
    blocks.  One more token either starts a new block (the last one is full) or, when the
    last block is partly filled and shared (count > 1), first replaces it by a fresh block
    (copy-on-write: the real engine copies the KV data too).  Forking shares every block
    (counts + 1); freeing drops the counts and returns blocks that reach 0 to the list.
  * Section "PagedAttention: block tables": copy-on-write happens when a sequence must write
    into a block whose count is above 1; only that block is copied.
  * Section "Chunked prefill": a step's token budget is filled with one token per running
    decode first, then with a chunk of a pending prefill; a 10,000-token prompt with a
    ~1,500-token chunk takes about 7 steps.
  * transformers "Continuous batching architecture", section "Scheduler": three budgets
    (max_batch_tokens query tokens per step, the KV pages that exist, max_requests_per_batch
    requests per step); FIFO takes active decodes, then active prefills, then waiting
    requests in arrival order; PrefillFirst completes split prefills before resuming decode.
    Its "Chunked prefill" paragraph: a prompt that exceeds the remaining budget is processed
    as far as it fits and continued on later steps.

  * transformers "Continuous batching architecture", sections "Prefix caching" and "Eviction",
    and "LLM learning path 3.3", section "Prefix caching and RadixAttention" (hash-based
    blocks): a completed block is identified by a hash of its tokens together with the hash of
    every block before it; a new prompt reuses its longest run of leading cached blocks and
    skips their prefill; shared blocks are reference-counted; a freed block keeps its content
    and hash, and when blocks without content run out the most recently initialized one is
    demoted (hash dropped) and reused.

Readings where the pages leave a step open (each also listed in the design notes):
  * Multi-token growth (a prefill chunk) follows the one-token rule token by token, so at
    most its first token can trigger a copy.
  * PrefillFirst order: active prefills, then active decodes, then waiting requests.
  * The cache budget: a chunk is cut to the tokens the free blocks (and the table width) can
    hold; a decode that cannot get its slot waits for a later step.
  * A request of prompt P and N new tokens: its last prompt position gives the first token,
    each later token comes from a one-token decode step, so it is in the batch for
    ceil-chunks(P) + N - 1 steps and holds P + N - 1 tokens at the end; it is retired (blocks
    freed) at the start of the step after its last token.
  * A request admitted in a step is not admitted twice in that step (a prompt completed in the
    step decodes from the next one).
  * Prefix caching: the hash is 64-bit FNV-1a over the parent hash (8 bytes) and the block's
    token ids (4 bytes each, little-endian); a match is confirmed by comparing the tokens;
    only blocks made entirely of prompt tokens are cached (generated tokens have no ids here);
    a match leaves at least the last prompt token to compute; a block whose content is already
    cached elsewhere is not registered again; "initialized" = the time the block's hash was
    registered.
"""
from __future__ import annotations


class AllocatorError(Exception):
    pass


def blocks_for(n_tokens: int, bs: int) -> int:
    return -(-n_tokens // bs)


FNV_OFFSET, FNV_PRIME, MASK64 = 0xCBF29CE484222325, 0x100000001B3, (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a (Fowler, Noll, Vo): for each byte, xor it in, then multiply by the prime."""
    h = FNV_OFFSET
    for byte in data:
        h = ((h ^ byte) * FNV_PRIME) & MASK64
    return h


def block_hash(parent: int, tokens) -> int:
    """Chained content hash: FNV-1a over the parent hash's 8 bytes and each token id's 4 bytes
    (little-endian)."""
    return fnv1a64(int(parent).to_bytes(8, "little") + b"".join(
        (int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens))


class BlockAllocator:
    """Free list (take from the end), reference counts, block tables and token counts; with
    prefix caching, content hashes of full prompt blocks and the initialized free blocks."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 prefix_caching: bool = False):
        if num_blocks < 1 or block_size < 4 or max_blocks_per_seq < 1:
            raise AllocatorError("bad pool shape")
        self.bs = block_size
        self.max_blocks = max_blocks_per_seq
        self.free = list(range(num_blocks))      # blocks without cached content
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.prefix = prefix_caching
        self.hash_of: dict[int, int] = {}        # block -> content hash
        self.content: dict[int, tuple] = {}      # block -> (parent hash, token ids)
        self.born: dict[int, int] = {}           # block -> initialization order
        self.cache: dict[int, int] = {}          # content hash -> block
        self.idle: set[int] = set()              # free blocks that keep cached content
        self.clock = 0
        self.hashed: dict[int, tuple] = {}       # seq -> (blocks hashed, chain hash)

    def num_free(self) -> int:
        return len(self.free) + len(self.idle)

    def _take(self) -> int:
        if self.free:
            b = self.free.pop()
        elif self.idle:
            b = max(self.idle, key=lambda x: self.born[x])   # most recently initialized
            self.idle.discard(b)
            h = self.hash_of.pop(b)
            if self.cache.get(h) == b:
                del self.cache[h]
            del self.content[b], self.born[b]
        else:
            raise AllocatorError("out of blocks")
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.prefix and b in self.hash_of:
            self.idle.add(b)
        else:
            self.free.append(b)

    def add_seq_cached(self, seq: int, tokens) -> int:
        """New sequence starting from the longest cached chain of the prompt's full blocks."""
        if seq in self.tables or len(tokens) < 1:
            raise AllocatorError("bad sequence")
        table, chain = [], 0
        if self.prefix:
            for j in range(min((len(tokens) - 1) // self.bs, self.max_blocks)):
                blk = tuple(int(t) for t in tokens[j * self.bs:(j + 1) * self.bs])
                h = block_hash(chain, blk)
                b = self.cache.get(h)
                if b is None or self.content[b] != (chain, blk):
                    break
                if self.ref[b] == 0:
                    self.idle.discard(b)
                self.ref[b] += 1
                table.append(b)
                chain = h
        self.tables[seq] = table
        self.lens[seq] = len(table) * self.bs
        self.hashed[seq] = (len(table), chain)
        return self.lens[seq]

    def hash_blocks(self, seq: int, tokens, n_tokens: int) -> None:
        if not self.prefix:
            return
        done, chain = self.hashed.get(seq, (0, 0))
        for j in range(done, n_tokens // self.bs):
            b = self.tables[seq][j]
            blk = tuple(int(t) for t in tokens[j * self.bs:(j + 1) * self.bs])
            h = block_hash(chain, blk)
            if b not in self.hash_of and self.ref[b] == 1 and h not in self.cache:
                self.hash_of[b] = h
                self.content[b] = (chain, blk)
                self.clock += 1
                self.born[b] = self.clock
                self.cache[h] = b
            chain = h
            done = j + 1
        self.hashed[seq] = (done, chain)

    def needed(self, seq: int, n: int) -> int:
        """Blocks growing `seq` (or creating it) by n tokens would take from the free list."""
        if n <= 0:
            return 0
        if seq not in self.tables:
            return blocks_for(n, self.bs)
        table, length = self.tables[seq], self.lens[seq]
        count = 0
        shared_partial = length % self.bs != 0 and self.ref[table[-1]] > 1
        if shared_partial:
            count += 1
        count += blocks_for(length + n, self.bs) - len(table)
        return count

    def add_seq(self, seq: int, n_tokens: int) -> None:
        if seq in self.tables:
            raise AllocatorError("sequence exists")
        nb = blocks_for(n_tokens, self.bs)
        if nb > self.max_blocks or nb > self.num_free():
            raise AllocatorError("does not fit")
        self.tables[seq] = [self._take() for _ in range(nb)]
        self.lens[seq] = n_tokens

    def append(self, seq: int, n_tokens: int) -> list[tuple[int, int]]:
        """Grow seq by n_tokens, one token at a time; returns the (old, new) block copies."""
        if seq not in self.tables:
            raise AllocatorError("no such sequence")
        if blocks_for(self.lens[seq] + n_tokens, self.bs) > self.max_blocks:
            raise AllocatorError("table too narrow")
        if self.needed(seq, n_tokens) > self.num_free():
            raise AllocatorError("does not fit")
        copies = []
        table = self.tables[seq]
        for _ in range(n_tokens):
            length = self.lens[seq]
            if length % self.bs == 0:
                table.append(self._take())
            elif self.ref[table[-1]] > 1:
                old = table[-1]
                self.ref[old] -= 1
                table[-1] = self._take()
                copies.append((old, table[-1]))
            self.lens[seq] = length + 1
        return copies

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.tables or child in self.tables:
            raise AllocatorError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        self.hashed[child] = self.hashed.get(parent, (0, 0))
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self._release(b)
        del self.lens[seq]
        self.hashed.pop(seq, None)

    def fits(self, seq: int) -> int:
        """Most tokens seq (or a new sequence) can grow by with the free blocks and table width."""
        free = self.num_free()
        if seq not in self.tables:
            return min(free, self.max_blocks) * self.bs
        table, length = self.tables[seq], self.lens[seq]
        slack = len(table) * self.bs - length
        if slack > 0 and self.ref[table[-1]] > 1:
            free -= 1
            if free < 0:
                return 0
        return slack + min(free, self.max_blocks - len(table)) * self.bs


WAITING, PREFILL, DECODE, DONE = "waiting", "prefill", "decode", "done"


class Request:
    def __init__(self, rid: int, prompt: int, max_new: int, tokens=None):
        self.id, self.prompt, self.max_new = rid, prompt, max_new
        self.tokens = None if tokens is None else [int(t) for t in tokens]
        self.done = 0          # prompt tokens in the cache
        self.generated = 0     # tokens produced
        self.state = WAITING


class Scheduler:
    """FIFO or PrefillFirst under max_batch_tokens, max_requests_per_batch and the free blocks."""

    def __init__(self, alloc: BlockAllocator, max_batch_tokens: int, max_requests_per_batch: int,
                 policy: str = "fifo"):
        if policy not in ("fifo", "prefill_first"):
            raise ValueError(policy)
        self.alloc = alloc
        self.max_tokens = max_batch_tokens
        self.max_reqs = max_requests_per_batch
        self.policy = policy
        self.requests: list[Request] = []   # arrival order; forks join at the end

    def add_request(self, rid: int, prompt: int, max_new: int, tokens=None) -> None:
        if any(r.id == rid for r in self.requests) or prompt < 1 or max_new < 1:
            raise AllocatorError("bad request")
        if blocks_for(prompt + max_new - 1, self.alloc.bs) > self.alloc.max_blocks:
            raise AllocatorError("request longer than a block table")
        self.requests.append(Request(rid, prompt, max_new, tokens))

    def fork_request(self, parent: int, child: int, max_new: int) -> None:
        p = next(r for r in self.requests if r.id == parent)
        if p.state != DECODE or max_new < p.generated:
            raise AllocatorError("bad fork")
        self.alloc.fork(parent, child)
        c = Request(child, p.prompt, max_new)
        c.done, c.generated, c.state = p.done, p.generated, DECODE
        self.requests.append(c)

    def step(self) -> dict:
        """One step: retire, admit in policy order, advance.  Returns the batch description."""
        finished = 0
        for r in self.requests:
            if r.state != DONE and r.generated >= r.max_new:
                if r.id in self.alloc.tables:
                    self.alloc.free_seq(r.id)
                r.state = DONE
                finished += 1
        batch = {"seq_ids": [], "q_lens": [], "kv_lens": [], "tables": [], "copies": [],
                 "num_decode": 0, "finished": finished, "cached": 0}
        budget = self.max_tokens
        start_state = {r.id: r.state for r in self.requests}

        def admit(r: Request, n: int) -> None:
            nonlocal budget
            if r.id not in self.alloc.tables:
                self.alloc.add_seq(r.id, n)
            else:
                batch["copies"] += self.alloc.append(r.id, n)
            batch["seq_ids"].append(r.id)
            batch["q_lens"].append(n)
            batch["kv_lens"].append(self.alloc.lens[r.id])
            batch["tables"].append(list(self.alloc.tables[r.id]))
            budget -= n
            if r.state == DECODE:
                batch["num_decode"] += 1
                r.generated += 1
            else:
                r.done += n
                r.state = PREFILL
                if self.alloc.prefix and r.tokens is not None:
                    self.alloc.hash_blocks(r.id, r.tokens, r.done)
                if r.done == r.prompt:
                    r.state = DECODE
                    r.generated = 1

        def take(kind: str) -> None:
            for r in self.requests:
                if len(batch["seq_ids"]) >= self.max_reqs or budget <= 0:
                    return
                if start_state[r.id] != kind or r.state != kind:
                    continue
                if kind == DECODE:
                    if self.alloc.needed(r.id, 1) <= self.alloc.num_free():
                        admit(r, 1)
                elif kind == WAITING and self.alloc.prefix and r.tokens is not None:
                    cached = self.alloc.add_seq_cached(r.id, r.tokens)
                    r.done = cached
                    n = min(r.prompt - r.done, budget, self.alloc.fits(r.id))
                    if n > 0:
                        batch["cached"] += cached
                        admit(r, n)
                    else:
                        self.alloc.free_seq(r.id)
                        r.done = 0
                else:
                    n = min(r.prompt - r.done, budget, self.alloc.fits(r.id))
                    if n > 0:
                        admit(r, n)

        order = (DECODE, PREFILL, WAITING) if self.policy == "fifo" else (PREFILL, DECODE, WAITING)
        for kind in order:
            take(kind)
        return batch

    def num_active(self) -> int:
        return sum(r.state != DONE for r in self.requests)
