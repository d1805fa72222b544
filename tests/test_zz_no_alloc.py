"""cb_ragged_paged_attention_noalloc: the attention entry point for callers that cannot allocate
device memory (no scratch allocator offered to them, or no cudaMalloc allowed in their running
loop).  Its scratch is a fixed array inside the library.  Called here through the C ABI and
compared with the regular entry point, which takes a caller-allocated workspace, on two calls
in a row (the second call reuses the scratch the first one left behind)."""
import ctypes

import numpy as np
import pytest
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from gpu_util import ATOL, RTOL, DeviceBatch, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(lib, db, out, lse):
    b = db.b
    dims = cb.CbDims(b.num_seqs, b.num_tokens, b.num_q_heads, b.num_kv_heads, b.head_dim,
                     b.num_pages, b.max_blocks)
    st = lib.cb_ragged_paged_attention_noalloc(
        db.q.data_ptr(), db.k_pages.data_ptr(), db.v_pages.data_ptr(), db.block_table.data_ptr(),
        db.cu.data_ptr(), db.kv_lens.data_ptr(), b.block_size, b.scale, out.data_ptr(),
        lse.data_ptr(), ctypes.byref(dims), torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("which", ["mixed-small", "decode-split"])
def test_noalloc_matches_regular_entry_point_twice(cuda_lib, which):
    if which == "mixed-small":
        b = workloads.build_batch([1, 40, 0, 1, 129, 1], [33, 40, 12, 500, 329, 1], 8, 2, 128,
                                  32, seed=901)
    else:  # decode sequences cut across many CTAs, so the scratch holds partial results
        b = workloads.build_batch([1] * 6, [3000, 17, 800, 4096, 1, 2500], 32, 8, 128, 32,
                                  seed=902)
    db = DeviceBatch(b)
    db.append()
    ref_out, ref_lse = db.attend(lse=True)
    assert cb.get_device_error() == cb.CB_OK
    lib = cb.library()
    for _ in range(2):
        out = torch.full_like(db.q, float("nan"))
        lse = torch.full((b.num_tokens, b.num_q_heads), float("nan"), dtype=torch.float32,
                         device="cuda")
        st = _noalloc(lib, db, out, lse)
        assert st == cb.CB_OK, lib.cb_last_error_message()
        assert cb.get_device_error() == cb.CB_OK
        assert_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy().astype(np.float64),
                     "noalloc out", atol=ATOL, rtol=RTOL)
        assert_close(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64),
                     "noalloc lse", atol=1e-3, rtol=1e-3)


def test_noalloc_rejects_batches_beyond_its_scratch(cuda_lib):
    lib = cb.library()
    # 4096 sequences x 128 query heads x head_dim 128 needs far more than the built-in scratch
    dims = cb.CbDims(4096, 4096, 128, 8, 128, 100000, 64)
    need = lib.cb_attention_workspace_size(ctypes.byref(dims), 16)
    assert need > 32 * 1024 * 1024
    p = ctypes.c_void_p(256)
    st = lib.cb_ragged_paged_attention_noalloc(p, p, p, p, p, p, 16, 0.125, p, None,
                                               ctypes.byref(dims), None)
    assert st == cb.CB_ERR_UNSUPPORTED
    assert b"scratch" in lib.cb_last_error_message()
