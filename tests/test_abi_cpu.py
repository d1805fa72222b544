"""The C ABI library builds, loads without a GPU, exports every symbol the header declares,
and rejects bad host-side arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import continuous_batching_paged_gb300 as cb
from continuous_batching_paged_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return cb.library()


def header_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(cb_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("cb_kv_append", "cb_ragged_paged_attention", "cb_attention_workspace_size",
                     "cb_get_device_error", "cb_status_string", "cb_copy_blocks", "cb_kv_offload",
                     "cb_kv_restore", "cb_alloc_create", "cb_sched_step"):
        assert required in names


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert cb.status_string(cb.CB_OK) == "CB_OK"
    assert cb.status_string(cb.CB_ERR_OUT_OF_RANGE) == "CB_ERR_OUT_OF_RANGE"
    assert cb.status_string(99) == "CB_ERR_UNKNOWN"
    assert lib.cb_version() >= 100


def _dims(**kw):
    base = dict(num_seqs=4, num_tokens=35, num_q_heads=4, num_kv_heads=2, head_dim=64,
                num_pages=24, max_blocks_per_seq=9)
    base.update(kw)
    return cb.CbDims(**base)


def test_workspace_size_is_host_arithmetic(lib):
    n = lib.cb_attention_workspace_size(ctypes.byref(_dims()))
    assert n > 0 and n % 256 == 0
    # grows with the number of sequences, heads and tokens (the chunk-unit order), never with
    # the pool or the table width
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(num_seqs=400))) > n
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(num_q_heads=8))) > n
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(num_pages=999))) == n
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(max_blocks_per_seq=999))) == n
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(num_tokens=999999))) > n
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(head_dim=96))) == 0
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(num_q_heads=3))) == 0  # 3 % 2
    assert lib.cb_attention_workspace_size(ctypes.byref(_dims(num_seqs=-1))) == 0
    assert lib.cb_attention_workspace_size(None) == 0


def _append_status(lib, dims, block_size, ptr=16):
    p = ctypes.c_void_p(ptr)
    return lib.cb_kv_append(p, p, p, p, p, p, p, block_size, ctypes.byref(dims), None)


def test_host_validation_rejects_before_cuda(lib):
    assert _append_status(lib, _dims(), 3) == cb.CB_ERR_INVALID_ARG
    assert b"at least 4" in lib.cb_last_error_message()
    assert _append_status(lib, _dims(num_q_heads=5), 16) == cb.CB_ERR_INVALID_ARG
    assert _append_status(lib, _dims(head_dim=80), 16) == cb.CB_ERR_UNSUPPORTED
    assert _append_status(lib, _dims(num_pages=0), 16) == cb.CB_ERR_INVALID_ARG
    assert _append_status(lib, _dims(), 16, ptr=24) == cb.CB_ERR_INVALID_ARG   # misaligned
    assert b"16-byte" in lib.cb_last_error_message()
    # an empty batch is a valid no-op
    assert _append_status(lib, _dims(num_tokens=0, num_seqs=0), 16) == cb.CB_OK
    p = ctypes.c_void_p(256)
    dims = _dims()
    # workspace too small -> rejected before any launch
    st = lib.cb_ragged_paged_attention(p, p, p, p, p, p, 16, 0.125, p, None, p, 256,
                                       ctypes.byref(dims), None)
    assert st == cb.CB_ERR_INVALID_ARG and b"workspace" in lib.cb_last_error_message()
    st = lib.cb_ragged_paged_attention(p, p, p, p, p, p, 16, -1.0, p, None, p, 1 << 30,
                                       ctypes.byref(dims), None)
    assert st == cb.CB_ERR_INVALID_ARG and b"scale" in lib.cb_last_error_message()
    st = lib.cb_ragged_paged_attention(p, p, p, p, None, p, 16, 0.125, p, None, p, 1 << 30,
                                       ctypes.byref(dims), None)
    assert st == cb.CB_ERR_INVALID_ARG and b"null" in lib.cb_last_error_message()


def test_new_entries_validate_on_the_host(lib):
    # the one-call step and the pass time stamps reject bad arguments before any CUDA call
    p = ctypes.c_void_p(256)
    dims = _dims()
    st = lib.cb_append_attention(None, p, p, p, p, p, p, p, 16, 0.125, p, None, p, 1 << 30,
                                 ctypes.byref(dims), None, None)
    assert st == cb.CB_ERR_INVALID_ARG and b"null" in lib.cb_last_error_message()
    st = lib.cb_append_attention(ctypes.c_void_p(264), p, p, p, p, p, p, p, 16, 0.125, p, None,
                                 p, 1 << 30, ctypes.byref(dims), None, None)
    assert st == cb.CB_ERR_INVALID_ARG and b"16-byte" in lib.cb_last_error_message()
    st = lib.cb_append_attention(p, p, p, p, p, p, p, p, 3, 0.125, p, None, p, 1 << 30,
                                 ctypes.byref(dims), None, None)
    assert st == cb.CB_ERR_INVALID_ARG and b"at least 4" in lib.cb_last_error_message()
    ts = (ctypes.c_uint64 * 4)()
    assert lib.cb_pass_timestamps(None, ts, None) == cb.CB_ERR_INVALID_ARG
    assert lib.cb_pass_timestamps(p, None, None) == cb.CB_ERR_INVALID_ARG


def test_build_flags_target_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)
