"""Host runtime of libcb (include/cb_sched.h): the paged-KV block allocator and the
continuous-batching scheduler, as thin ctypes wrappers over the library's C++ objects.

    alloc = BlockAllocator(num_blocks=4096, block_size=32, max_blocks_per_seq=256)
    sched = Scheduler(alloc, max_batch_tokens=2048, max_requests_per_batch=256, policy="fifo")
    sched.add_request(0, prompt_len=1000, max_new_tokens=300)
    step = sched.step()          # numpy views: cu_seqlens_q, kv_lens, block_table, copies
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import CbError, CB_OK, library

_I32P = ctypes.POINTER(ctypes.c_int32)
_POLICIES = {"fifo": 0, "prefill_first": 1}


class _Batch(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_cow", ctypes.c_int32), ("num_decode", ctypes.c_int32),
                ("num_finished", ctypes.c_int32), ("num_cached", ctypes.c_int32),
                ("cap_seqs", ctypes.c_int32),
                ("cap_cow", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("seq_ids", _I32P), ("cu_seqlens_q", _I32P), ("kv_lens", _I32P),
                ("block_table", _I32P), ("cow_src", _I32P), ("cow_dst", _I32P)]


class _SchedConfig(ctypes.Structure):
    _fields_ = [("max_batch_tokens", ctypes.c_int32), ("max_requests_per_batch", ctypes.c_int32),
                ("policy", ctypes.c_int32)]


_declared = False


def _lib() -> ctypes.CDLL:
    global _declared
    lib = library()
    if not _declared:
        P, I = ctypes.c_void_p, ctypes.c_int32
        lib.cb_alloc_create.restype = ctypes.c_int
        lib.cb_alloc_create.argtypes = [I, I, I, ctypes.POINTER(P)]
        lib.cb_alloc_destroy.restype = None
        lib.cb_alloc_destroy.argtypes = [P]
        lib.cb_alloc_add_seq.restype = ctypes.c_int
        lib.cb_alloc_add_seq.argtypes = [P, I, I]
        lib.cb_alloc_append.restype = ctypes.c_int
        lib.cb_alloc_append.argtypes = [P, I, I, _I32P, _I32P, _I32P]
        lib.cb_alloc_blocks_needed.restype = I
        lib.cb_alloc_blocks_needed.argtypes = [P, I, I]
        lib.cb_alloc_fork.restype = ctypes.c_int
        lib.cb_alloc_fork.argtypes = [P, I, I]
        lib.cb_alloc_free_seq.restype = ctypes.c_int
        lib.cb_alloc_free_seq.argtypes = [P, I]
        lib.cb_alloc_num_free.restype = I
        lib.cb_alloc_num_free.argtypes = [P]
        lib.cb_alloc_ref_count.restype = I
        lib.cb_alloc_ref_count.argtypes = [P, I]
        lib.cb_alloc_table.restype = ctypes.c_int
        lib.cb_alloc_table.argtypes = [P, I, _I32P, I, _I32P, _I32P]
        lib.cb_sched_create.restype = ctypes.c_int
        lib.cb_sched_create.argtypes = [P, ctypes.POINTER(_SchedConfig), ctypes.POINTER(P)]
        lib.cb_sched_destroy.restype = None
        lib.cb_sched_destroy.argtypes = [P]
        lib.cb_sched_add_request.restype = ctypes.c_int
        lib.cb_sched_add_request.argtypes = [P, I, I, I]
        lib.cb_alloc_set_prefix_caching.restype = ctypes.c_int
        lib.cb_alloc_set_prefix_caching.argtypes = [P, I]
        lib.cb_alloc_add_seq_cached.restype = ctypes.c_int
        lib.cb_alloc_add_seq_cached.argtypes = [P, I, _I32P, I, _I32P]
        lib.cb_alloc_hash_blocks.restype = ctypes.c_int
        lib.cb_alloc_hash_blocks.argtypes = [P, I, _I32P, I]
        lib.cb_alloc_num_cached.restype = I
        lib.cb_alloc_num_cached.argtypes = [P]
        lib.cb_sched_add_request_tokens.restype = ctypes.c_int
        lib.cb_sched_add_request_tokens.argtypes = [P, I, _I32P, I, I]
        lib.cb_sched_fork_request.restype = ctypes.c_int
        lib.cb_sched_fork_request.argtypes = [P, I, I, I]
        lib.cb_sched_step.restype = ctypes.c_int
        lib.cb_sched_step.argtypes = [P, ctypes.POINTER(_Batch)]
        lib.cb_sched_num_active.restype = I
        lib.cb_sched_num_active.argtypes = [P]
        _declared = True
    return lib


def _check(st: int, where: str) -> None:
    if st != CB_OK:
        raise CbError(st, where, _lib().cb_last_error_message().decode())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


class BlockAllocator:
    """Free stack of physical blocks, reference counts, per-sequence block tables."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self._h = ctypes.c_void_p()
        _check(_lib().cb_alloc_create(num_blocks, block_size, max_blocks_per_seq,
                                      ctypes.byref(self._h)), "cb_alloc_create")
        self.block_size = block_size
        self.max_blocks = max_blocks_per_seq

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib().cb_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def add_seq(self, seq: int, n_tokens: int) -> None:
        _check(_lib().cb_alloc_add_seq(self._h, seq, n_tokens), "cb_alloc_add_seq")

    def append(self, seq: int, n_tokens: int) -> list[tuple[int, int]]:
        src, dst, n = ctypes.c_int32(-1), ctypes.c_int32(-1), ctypes.c_int32(0)
        _check(_lib().cb_alloc_append(self._h, seq, n_tokens, ctypes.byref(src),
                                      ctypes.byref(dst), ctypes.byref(n)), "cb_alloc_append")
        return [(src.value, dst.value)] if n.value else []

    def blocks_needed(self, seq: int, n_tokens: int) -> int:
        return int(_lib().cb_alloc_blocks_needed(self._h, seq, n_tokens))

    def fork(self, parent: int, child: int) -> None:
        _check(_lib().cb_alloc_fork(self._h, parent, child), "cb_alloc_fork")

    def free_seq(self, seq: int) -> None:
        _check(_lib().cb_alloc_free_seq(self._h, seq), "cb_alloc_free_seq")

    def set_prefix_caching(self, enable: bool = True) -> None:
        _check(_lib().cb_alloc_set_prefix_caching(self._h, int(enable)), "cb_alloc_set_prefix_caching")

    def add_seq_cached(self, seq: int, tokens) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int32()
        _check(_lib().cb_alloc_add_seq_cached(self._h, seq, _ptr(t), t.size, ctypes.byref(n)),
               "cb_alloc_add_seq_cached")
        return n.value

    def hash_blocks(self, seq: int, tokens) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(_lib().cb_alloc_hash_blocks(self._h, seq, _ptr(t), t.size), "cb_alloc_hash_blocks")

    def num_cached(self) -> int:
        return int(_lib().cb_alloc_num_cached(self._h))

    def num_free(self) -> int:
        return int(_lib().cb_alloc_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(_lib().cb_alloc_ref_count(self._h, block))

    def table(self, seq: int) -> tuple[list[int], int]:
        buf = np.empty(self.max_blocks, dtype=np.int32)
        nb, nt = ctypes.c_int32(), ctypes.c_int32()
        _check(_lib().cb_alloc_table(self._h, seq, _ptr(buf), self.max_blocks, ctypes.byref(nb),
                                     ctypes.byref(nt)), "cb_alloc_table")
        return buf[:nb.value].tolist(), nt.value


class Scheduler:
    """FIFO or PrefillFirst continuous-batching scheduler over a BlockAllocator."""

    def __init__(self, alloc: BlockAllocator, max_batch_tokens: int,
                 max_requests_per_batch: int, policy: str = "fifo"):
        self.alloc = alloc  # keeps the allocator alive
        cfg = _SchedConfig(max_batch_tokens, max_requests_per_batch, _POLICIES[policy])
        self._h = ctypes.c_void_p()
        _check(_lib().cb_sched_create(alloc._h, ctypes.byref(cfg), ctypes.byref(self._h)),
               "cb_sched_create")
        cap = max_requests_per_batch
        self._seq_ids = np.empty(cap, dtype=np.int32)
        self._cu = np.empty(cap + 1, dtype=np.int32)
        self._kv = np.empty(cap, dtype=np.int32)
        self._table = np.empty((cap, alloc.max_blocks), dtype=np.int32)
        self._src = np.empty(cap, dtype=np.int32)
        self._dst = np.empty(cap, dtype=np.int32)
        self._batch = _Batch(0, 0, 0, 0, 0, 0, cap, cap, alloc.max_blocks, _ptr(self._seq_ids),
                             _ptr(self._cu), _ptr(self._kv), _ptr(self._table), _ptr(self._src),
                             _ptr(self._dst))

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib().cb_sched_destroy(self._h)
            self._h = ctypes.c_void_p()

    def add_request(self, rid: int, prompt_len: int, max_new_tokens: int) -> None:
        _check(_lib().cb_sched_add_request(self._h, rid, prompt_len, max_new_tokens),
               "cb_sched_add_request")

    def add_request_tokens(self, rid: int, tokens, max_new_tokens: int) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(_lib().cb_sched_add_request_tokens(self._h, rid, _ptr(t), t.size, max_new_tokens),
               "cb_sched_add_request_tokens")

    def fork_request(self, parent: int, child: int, max_new_tokens: int) -> None:
        _check(_lib().cb_sched_fork_request(self._h, parent, child, max_new_tokens),
               "cb_sched_fork_request")

    def num_active(self) -> int:
        return int(_lib().cb_sched_num_active(self._h))

    def step(self) -> dict:
        """Build the next step.  The arrays are views into buffers the next call overwrites."""
        _check(_lib().cb_sched_step(self._h, ctypes.byref(self._batch)), "cb_sched_step")
        b = self._batch
        s, c = b.num_seqs, b.num_cow
        return {"seq_ids": self._seq_ids[:s], "cu_seqlens_q": self._cu[:s + 1],
                "kv_lens": self._kv[:s], "block_table": self._table[:s],
                "cow_src": self._src[:c], "cow_dst": self._dst[:c],
                "num_tokens": b.num_tokens, "num_decode": b.num_decode,
                "num_finished": b.num_finished, "num_cached": b.num_cached}
