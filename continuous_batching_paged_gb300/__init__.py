"""Ragged paged attention and paged KV-append for GB300 (sm_103a).

Thin ctypes binding of libcb (include/cb.h).  It only marshals arguments: every step of the
path runs in the library's CUDA kernels, and PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing or cannot be built, every call raises.

    import continuous_batching_paged_gb300 as cb
    cb.kv_append(k_new, v_new, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size)
    out = cb.ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                                    block_size, scale)
    cb.check_device_error()
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "CbError", "CB_OK", "CB_ERR_INVALID_ARG", "CB_ERR_UNSUPPORTED", "CB_ERR_OUT_OF_RANGE",
    "CB_ERR_TIMEOUT", "CB_ERR_CUDA", "CbDims", "CbOptions", "library", "library_path",
    "kv_append", "ragged_paged_attention", "workspace_size", "get_device_error",
    "check_device_error", "status_string", "copy_blocks", "kv_offload", "kv_restore",
    "append_attention", "selftest_wait_timeout",
]

CB_OK = 0
CB_ERR_INVALID_ARG = 1
CB_ERR_UNSUPPORTED = 2
CB_ERR_OUT_OF_RANGE = 3
CB_ERR_TIMEOUT = 4
CB_ERR_CUDA = 5

_PKG = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_PKG, "libcb.so")


class CbDims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32)]


NUM_PHASE_EVENTS = 5
OPT_SERIAL = 1


class CbOptions(ctypes.Structure):
    _fields_ = [("decode_ctas", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("phase_events", ctypes.POINTER(ctypes.c_void_p)),
                ("window", ctypes.c_int32), ("reserved32", ctypes.c_int32),
                ("reserved", ctypes.c_int64 * 3)]


class CbError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" + (f" ({detail})" if detail else ""))


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None

_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)


def _declare(lib: ctypes.CDLL) -> None:
    lib.cb_version.restype = ctypes.c_int32
    lib.cb_version.argtypes = []
    lib.cb_status_string.restype = ctypes.c_char_p
    lib.cb_status_string.argtypes = [ctypes.c_int]
    lib.cb_last_error_message.restype = ctypes.c_char_p
    lib.cb_last_error_message.argtypes = []
    lib.cb_attention_workspace_size.restype = ctypes.c_size_t
    lib.cb_attention_workspace_size.argtypes = [ctypes.POINTER(CbDims)]
    lib.cb_kv_append.restype = ctypes.c_int
    lib.cb_kv_append.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int32,
                                 ctypes.POINTER(CbDims), _P]
    attn = [_P, _P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_float, _P, _P, _P, ctypes.c_size_t,
            ctypes.POINTER(CbDims)]
    lib.cb_ragged_paged_attention.restype = ctypes.c_int
    lib.cb_ragged_paged_attention.argtypes = attn + [_P]
    lib.cb_ragged_paged_attention_ex.restype = ctypes.c_int
    lib.cb_ragged_paged_attention_ex.argtypes = attn + [ctypes.POINTER(CbOptions), _P]
    lib.cb_append_attention.restype = ctypes.c_int
    lib.cb_append_attention.argtypes = [_P, _P, _P, _P] + [_P, _P, _P, _P, ctypes.c_int32,
                                                          ctypes.c_float, _P, _P, _P,
                                                          ctypes.c_size_t, ctypes.POINTER(CbDims),
                                                          ctypes.POINTER(CbOptions), _P]
    lib.cb_ragged_paged_attention_noalloc.restype = ctypes.c_int
    lib.cb_ragged_paged_attention_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_int32,
                                                      ctypes.c_float, _P, _P,
                                                      ctypes.POINTER(CbDims), _P]
    lib.cb_get_device_error.restype = ctypes.c_int
    lib.cb_get_device_error.argtypes = [_P]
    lib.cb_pass_timestamps.restype = ctypes.c_int
    lib.cb_pass_timestamps.argtypes = [_P, ctypes.POINTER(ctypes.c_uint64), _P]
    lib.cb_selftest_wait_timeout.restype = ctypes.c_int
    lib.cb_selftest_wait_timeout.argtypes = [ctypes.c_int32, _P, _P]
    lib.cb_copy_blocks.restype = ctypes.c_int
    lib.cb_copy_blocks.argtypes = [_P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.POINTER(CbDims), _P]
    lib.cb_kv_offload.restype = ctypes.c_int
    lib.cb_kv_offload.argtypes = [_P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.POINTER(CbDims), _P, _P, _P]
    lib.cb_kv_restore.restype = ctypes.c_int
    lib.cb_kv_restore.argtypes = [_P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.POINTER(CbDims), _P, _P, _P]


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded libcb (built in-tree first if it is missing or older than its sources)."""
    global _lib
    with _lock:
        if _lib is None:
            from . import _build
            path = library_path()
            if build_if_missing and _build.is_stale():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libcb is not built ({path}); run the package build first")
            lib = ctypes.CDLL(path)
            _declare(lib)
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    return library().cb_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != CB_OK:
        detail = library().cb_last_error_message().decode()
        raise CbError(status, where, detail)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _dims(T, S, Hq, Hkv, D, P, MB) -> CbDims:
    return CbDims(int(S), int(T), int(Hq), int(Hkv), int(D), int(P), int(MB))


def _check_meta(block_table, cu_seqlens_q, kv_lens):
    import torch
    for name, t in (("block_table", block_table), ("cu_seqlens_q", cu_seqlens_q),
                    ("kv_lens", kv_lens)):
        _require(t.dtype == torch.int32, f"{name} must be int32")
        _require(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _require(block_table.dim() == 2, "block_table must be [num_seqs, max_blocks]")
    S = kv_lens.numel()
    _require(cu_seqlens_q.numel() == S + 1, "cu_seqlens_q must have num_seqs + 1 entries")
    _require(block_table.shape[0] == S, "block_table must have num_seqs rows")
    return S


def _check_bf16(name, t, ndim):
    import torch
    _require(t.dtype == torch.bfloat16, f"{name} must be bfloat16")
    _require(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _require(t.dim() == ndim, f"{name} must have {ndim} dimensions")


def _pool_dims(k_pages, v_pages, block_size) -> CbDims:
    _check_bf16("k_pages", k_pages, 4)
    _require(k_pages.shape == v_pages.shape, "v_pages must match k_pages")
    P, bs, Hkv, D = k_pages.shape
    _require(bs == block_size, "k_pages.shape[1] must be block_size")
    return _dims(0, 0, Hkv, Hkv, D, P, 1)


def _check_ids(name, t):
    import torch
    _require(t.dtype == torch.int32 and t.is_cuda and t.is_contiguous(),
             f"{name} must be a contiguous int32 CUDA tensor")


def selftest_wait_timeout(limit_us: int, waited_ns=None, stream=None) -> None:
    """Launch one GPU wait that nothing completes; it gives up after limit_us and records
    CB_ERR_TIMEOUT for get_device_error() (cb_selftest_wait_timeout)."""
    _check(library().cb_selftest_wait_timeout(int(limit_us), _ptr(waited_ns), _stream(stream)),
           "cb_selftest_wait_timeout")


def copy_blocks(k_pages, v_pages, src, dst, block_size, stream=None) -> None:
    """Block dst[i] of both pools receives block src[i] (cb_copy_blocks: copy-on-write data)."""
    dims = _pool_dims(k_pages, v_pages, block_size)
    _check_ids("src", src)
    _check_ids("dst", dst)
    _require(src.numel() == dst.numel(), "src and dst must have the same length")
    _check(library().cb_copy_blocks(_ptr(k_pages), _ptr(v_pages), _ptr(src), _ptr(dst),
                                    src.numel(), int(block_size), ctypes.byref(dims),
                                    _stream(stream)), "cb_copy_blocks")


def kv_offload(k_pages, v_pages, blocks, block_size, host_k, host_v, stream=None) -> None:
    """Gather blocks of both pools into pinned host tensors [n, bs, Hkv, D] (cb_kv_offload)."""
    dims = _pool_dims(k_pages, v_pages, block_size)
    _check_ids("blocks", blocks)
    n = blocks.numel()
    for name, h in (("host_k", host_k), ("host_v", host_v)):
        _require(h.is_pinned() and h.is_contiguous() and h.numel() * h.element_size()
                 >= n * k_pages[0].numel() * 2, f"{name} must be pinned, contiguous, large enough")
    _check(library().cb_kv_offload(_ptr(k_pages), _ptr(v_pages), _ptr(blocks), n,
                                   int(block_size), ctypes.byref(dims), _ptr(host_k),
                                   _ptr(host_v), _stream(stream)), "cb_kv_offload")


def kv_restore(k_pages, v_pages, blocks, block_size, host_k, host_v, stream=None) -> None:
    """Scatter pinned host tensors [n, bs, Hkv, D] into blocks of both pools (cb_kv_restore)."""
    dims = _pool_dims(k_pages, v_pages, block_size)
    _check_ids("blocks", blocks)
    n = blocks.numel()
    for name, h in (("host_k", host_k), ("host_v", host_v)):
        _require(h.is_pinned() and h.is_contiguous() and h.numel() * h.element_size()
                 >= n * k_pages[0].numel() * 2, f"{name} must be pinned, contiguous, large enough")
    _check(library().cb_kv_restore(_ptr(k_pages), _ptr(v_pages), _ptr(blocks), n,
                                   int(block_size), ctypes.byref(dims), _ptr(host_k),
                                   _ptr(host_v), _stream(stream)), "cb_kv_restore")


def kv_append(k_new, v_new, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size,
              stream=None) -> None:
    """Scatter k_new/v_new [T, Hkv, D] into k_pages/v_pages [P, bs, Hkv, D] (cb_kv_append)."""
    _check_bf16("k_new", k_new, 3)
    _check_bf16("v_new", v_new, 3)
    _check_bf16("k_pages", k_pages, 4)
    _check_bf16("v_pages", v_pages, 4)
    S = _check_meta(block_table, cu_seqlens_q, kv_lens)
    T, Hkv, D = k_new.shape
    _require(tuple(v_new.shape) == (T, Hkv, D), "v_new must match k_new")
    _require(tuple(k_pages.shape[1:]) == (block_size, Hkv, D), "k_pages must be [P, bs, Hkv, D]")
    _require(k_pages.shape == v_pages.shape, "v_pages must match k_pages")
    dims = _dims(T, S, Hkv, Hkv, D, k_pages.shape[0], block_table.shape[1])
    st = library().cb_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                                _ptr(block_table), _ptr(cu_seqlens_q), _ptr(kv_lens),
                                int(block_size), ctypes.byref(dims), _stream(stream))
    _check(st, "cb_kv_append")


def workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, num_tokens) -> int:
    """Bytes of device workspace an attention call on this batch shape needs
    (cb_attention_workspace_size; 0 for an invalid shape)."""
    dims = _dims(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, 1, 1)
    return int(library().cb_attention_workspace_size(ctypes.byref(dims)))


def ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size,
                           scale, out=None, lse=None, workspace=None, decode_ctas: int = 0,
                           phase_events=None, serial: bool = False, window: int = 0,
                           stream=None, k_new=None, v_new=None):
    """One attention pass over the ragged batch (cb_ragged_paged_attention_ex).

    q [T, Hq, D] bf16; pages [P, bs, Hkv, D] bf16 (after the append); returns out [T, Hq, D]
    bf16, or (out, lse) when ``lse`` is True or an fp32 [T, Hq] tensor.  ``phase_events``:
    optional sequence of NUM_PHASE_EVENTS recorded torch.cuda.Event objects; the call records
    them around its planner and its attention launch (see cb_options in cb.h).  ``serial``
    runs the decode pass and the chunk pass as two launches instead of one.  ``window`` > 0
    selects sliding-window attention over the last ``window`` keys of each query.
    """
    import torch
    _check_bf16("q", q, 3)
    _check_bf16("k_pages", k_pages, 4)
    _check_bf16("v_pages", v_pages, 4)
    S = _check_meta(block_table, cu_seqlens_q, kv_lens)
    T, Hq, D = q.shape
    P, bs, Hkv, D2 = k_pages.shape
    _require(bs == block_size and D2 == D, "k_pages must be [P, block_size, Hkv, D]")
    _require(k_pages.shape == v_pages.shape, "v_pages must match k_pages")
    if out is None:
        out = torch.empty_like(q)
    _check_bf16("out", out, 3)
    _require(tuple(out.shape) == (T, Hq, D), "out must be [T, Hq, D]")
    want_lse = lse is not None and lse is not False
    if lse is True:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    if lse is not None:
        _require(lse.dtype == torch.float32 and lse.is_contiguous() and tuple(lse.shape) == (T, Hq),
                 "lse must be a contiguous fp32 [T, Hq] tensor")
    dims = _dims(T, S, Hq, Hkv, D, P, block_table.shape[1])
    need = int(library().cb_attention_workspace_size(ctypes.byref(dims)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _require(workspace.dtype == torch.uint8 and workspace.is_contiguous(), "workspace must be uint8")
    opts = CbOptions(int(decode_ctas), OPT_SERIAL if serial else 0)
    opts.window = int(window)
    if phase_events is not None:
        _require(len(phase_events) == NUM_PHASE_EVENTS, f"need {NUM_PHASE_EVENTS} phase events")
        handles = (ctypes.c_void_p * NUM_PHASE_EVENTS)(*[int(e.cuda_event) for e in phase_events])
        _require(all(handles), "phase events must have been recorded once (created) before use")
        opts.phase_events = ctypes.cast(handles, ctypes.POINTER(ctypes.c_void_p))
    if k_new is None:
        st = library().cb_ragged_paged_attention_ex(
            _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(cu_seqlens_q),
            _ptr(kv_lens), int(block_size), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel(), ctypes.byref(dims), ctypes.byref(opts), _stream(stream))
        _check(st, "cb_ragged_paged_attention")
    else:
        _check_bf16("k_new", k_new, 3)
        _check_bf16("v_new", v_new, 3)
        _require(tuple(k_new.shape) == (T, Hkv, D) and k_new.shape == v_new.shape,
                 "k_new / v_new must be [T, Hkv, D]")
        st = library().cb_append_attention(
            _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages), _ptr(q), _ptr(block_table),
            _ptr(cu_seqlens_q), _ptr(kv_lens), int(block_size), float(scale), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel(), ctypes.byref(dims),
            ctypes.byref(opts), _stream(stream))
        _check(st, "cb_append_attention")
    return (out, lse) if want_lse else out


def append_attention(q, k_new, v_new, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                     block_size, scale, **kwargs):
    """kv_append then ragged_paged_attention in one call (cb_append_attention): same results,
    with the append and the attention planner in one launch.  Keyword arguments as for
    ragged_paged_attention."""
    return ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                                  block_size, scale, k_new=k_new, v_new=v_new, **kwargs)


def get_device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the device error word (a cb status)."""
    return int(library().cb_get_device_error(_stream(stream)))


def check_device_error(stream=None) -> None:
    _check(get_device_error(stream), "device")


def pass_timestamps(workspace, stream=None) -> tuple[int, int, int, int]:
    """%globaltimer stamps (ns) of the last attention call on `workspace`: first start and last
    end of the decode pass, then of the chunk pass (0, 0 for a pass without work).  Waits for
    the stream."""
    ts = (ctypes.c_uint64 * 4)()
    _check(library().cb_pass_timestamps(_ptr(workspace), ts, _stream(stream)), "cb_pass_timestamps")
    return tuple(int(x) for x in ts)
