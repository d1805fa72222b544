"""cb_ragged_paged_attention_noalloc: the attention entry point for callers that cannot allocate
device memory (no scratch allocator offered to them, or no cudaMalloc allowed in their running
loop).  Its scratch is a fixed array inside the library.  Called here through the C ABI on
batches of different shapes in turn, each compared bit for bit with the regular entry point
(which takes a caller-allocated workspace): both run the same kernels on the same plan, so
the scratch left behind by a call of another shape must change nothing."""
import ctypes

import pytest
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from gpu_util import DeviceBatch

pytestmark = pytest.mark.gpu


def _noalloc(lib, db, out, lse):
    b = db.b
    dims = cb.CbDims(b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads, b.head_dim,
                     b.num_pages, b.max_blocks)
    return lib.cb_ragged_paged_attention_noalloc(
        db.q.data_ptr(), db.k_pages.data_ptr(), db.v_pages.data_ptr(), db.block_table.data_ptr(),
        db.cu.data_ptr(), db.kv_lens.data_ptr(), b.block_size, b.scale, out.data_ptr(),
        lse.data_ptr(), ctypes.byref(dims), torch.cuda.current_stream().cuda_stream)


def _batches():
    # decode sequences cut across many CTAs (the scratch holds partial results and merge
    # counters), and a small mixed batch (chunks and decodes, another plan layout)
    split = workloads.build_batch([1] * 6, [3000, 17, 800, 4096, 1, 2500], 32, 8, 128, 32,
                                  seed=902, name="decode-split")
    mixed = workloads.build_batch([1, 40, 0, 1, 129, 1], [33, 40, 12, 500, 329, 1], 8, 2, 128,
                                  32, seed=901, name="mixed-small")
    return split, mixed


def test_noalloc_equals_regular_entry_point_across_shapes(cuda_lib):
    lib = cb.library()
    refs = []
    for b in _batches():
        db = DeviceBatch(b)
        db.append()
        out, lse = db.attend(lse=True)
        assert cb.get_device_error() == cb.CB_OK
        refs.append((db, out, lse))
    # decode-split, mixed-small, decode-split, mixed-small: every call finds the scratch the
    # call before it (of the other shape) left behind
    for i in (0, 1, 0, 1):
        db, ref_out, ref_lse = refs[i]
        out = torch.full_like(db.q, float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(lib, db, out, lse)
        assert st == cb.CB_OK, lib.cb_last_error_message()
        assert cb.get_device_error() == cb.CB_OK
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), db.b.name
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), db.b.name


def test_noalloc_rejects_batches_beyond_its_scratch(cuda_lib):
    lib = cb.library()
    # 4096 sequences x 128 query heads x head_dim 128 needs far more than the built-in scratch
    dims = cb.CbDims(4096, 4096, 128, 8, 128, 100000, 64)
    need = lib.cb_attention_workspace_size(ctypes.byref(dims))
    assert need > 32 * 1024 * 1024
    p = ctypes.c_void_p(256)
    st = lib.cb_ragged_paged_attention_noalloc(p, p, p, p, p, p, 16, 0.125, p, None,
                                               ctypes.byref(dims), None)
    assert st == cb.CB_ERR_UNSUPPORTED
    assert b"scratch" in lib.cb_last_error_message()
