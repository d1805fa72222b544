"""Helpers shared by the GPU parity tests: move a seeded batch to the device, run the CUDA path
through the C ABI, and compare with the oracle."""
from __future__ import annotations

import functools

import numpy as np
import torch

import continuous_batching_paged_gb300 as cb
import workloads
from oracle import paged_attention as opa

# Attention tolerance: elementwise |gpu - ref| <= ATOL + RTOL * |ref| (bf16 in, fp32 accumulate,
# bf16 out): max abs error 2e-2 plus 1e-2 relative, fixed for this bf16-in / fp32-accumulate path.
ATOL = 2e-2
RTOL = 1e-2


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class DeviceBatch:
    def __init__(self, b: workloads.Batch):
        self.b = b
        self.q = bf16_tensor(b.q)
        self.k_new = bf16_tensor(b.k_new)
        self.v_new = bf16_tensor(b.v_new)
        self.k_pages = bf16_tensor(b.k_pages)
        self.v_pages = bf16_tensor(b.v_pages)
        self.block_table = i32(b.block_table)
        self.cu = i32(b.cu_seqlens_q)
        self.kv_lens = i32(b.kv_lens)

    def append(self):
        cb.kv_append(self.k_new, self.v_new, self.k_pages, self.v_pages, self.block_table,
                     self.cu, self.kv_lens, self.b.block_size)

    def attend(self, lse=False, decode_ctas=0, block_table=None, k_pages=None, v_pages=None):
        # Workspace filled with 0xFF bytes (NaN as fp32): a read of a partial result that was
        # never written shows up as NaN in the output.
        ws = torch.full((cb.workspace_size(self.b.num_seqs, self.b.num_q_heads,
                                           self.b.num_kv_heads, self.b.head_dim,
                                           self.b.num_tokens),), 255,
                                           dtype=torch.uint8,
                        device="cuda")
        return cb.ragged_paged_attention(workspace=ws, *(
            self.q, self.k_pages if k_pages is None else k_pages,
            self.v_pages if v_pages is None else v_pages,
            self.block_table if block_table is None else block_table, self.cu, self.kv_lens,
            self.b.block_size, self.b.scale), lse=lse, decode_ctas=decode_ctas)


@functools.lru_cache(maxsize=5)
def named_config(n: int) -> workloads.Batch:
    """Named workload n, drawn once per test session (the large ones take a while)."""
    return workloads.make_config(n)


def oracle_append(b: workloads.Batch):
    return opa.kv_append(b.k_new, b.v_new, b.k_pages, b.v_pages, b.block_table, b.cu_seqlens_q,
                         b.kv_lens, b.block_size)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite values in the CUDA output"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        rel = float((err / np.maximum(np.abs(ref), 1e-6)).max())
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                             f"{atol} + {rtol}*|ref|; max abs err {err.max():.4g}, max rel err "
                             f"{rel:.4g}; first {idx}")
    return float(err.max()) if err.size else 0.0
