#!/usr/bin/env python
"""Benchmark of the ragged paged-attention hot path on GB300.

One step = one pass of the whole path over one synthetic batch: the paged KV-append and the
ragged paged-attention pass (cb_append_attention: append + planner in one launch, then the
attention kernel, whose CTAs run the split-KV decode pass with its LSE merge and the tcgen05
chunk pass).  Default workload: the mixed ragged
batch at max_batch_tokens = 2048 (120 decode tokens at prior context U[256, 8192] plus one
1928-token chunk at prior context 3000; 32 query / 8 KV heads, head_dim 128, block size 32), the
one batch of the named set in which every step of the path runs.

Prints ONE JSON line.  `value` is query tokens per second of the whole job, from device time
(CUDA events on the launching stream) with inputs resident in HBM; L2 is flushed (a 512 MiB
write, then a 512 MiB read) before every timed step.  `e2e` is the same metric through the Python API with the step's
inputs copied from pinned host memory and the output copied back inside the timed region.
`roofline` is the attention kernel's algorithmic bytes (or FLOPs, by the bound of the pass with
the larger ideal time) per launch over its average device time, measured by events the library
records around the launch.  `cpu_baseline` is the
float64 oracle timed on a bounded sample of the same workload on this host's cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixed|decode|prefill|longtail]
    python bench.py --impl reference ...     # the oracle as the reference arm
Multi-GPU (torchrun): each rank runs an independent replica (the path shards by sequence with no
exchange), timing is the max over ranks, and `value` sums all ranks' tokens ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged-attn decode KV GB/s (% of HBM peak); mixed-batch query tokens/sec"
WORKLOADS = {"tiny": 1, "decode": 2, "mixed": 3, "prefill": 4, "longtail": 5}
NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["cb", "reference"], default="cb")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="mixed")
    p.add_argument("--decode-ctas", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", action="store_true",
                   help="measure the headline workload only (skip the further batches)")
    p.add_argument("--serial", action="store_true",
                   help="run the decode pass and the chunk pass as two launches, one after the other")
    p.add_argument("--mode", choices=["path", "blocks", "serve", "graphs"], default="path",
                   help="path: the attention hot path (default); blocks: KV block copy / "
                        "offload / restore kernels; serve: a scheduler-driven serving loop; "
                        "graphs: step latency eager vs CUDA-graph replay")
    p.add_argument("--policy", choices=["fifo", "prefill_first"], default="fifo")
    p.add_argument("--separate", action="store_true",
                   help="issue the append and the attention pass as two calls instead of "
                        "cb_append_attention")
    p.add_argument("--window", type=int, default=0,
                   help="sliding-window attention over the last W keys (0: full causal)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


# ----------------------------------------------------------------------------- workload facts

def decode_kv_bytes(b: workloads.Batch, window: int = 0):
    """Algorithmic HBM bytes of the decode pass: every distinct K/V row a decode token reads
    (shared prefix pages once), plus its q and out rows; and the same with sharing counted per
    sequence ("logical")."""
    q_lens = np.diff(b.cu_seqlens_q)
    row_bytes = b.num_kv_heads * b.head_dim * 2 * 2          # K + V, bf16
    slots = []
    logical = 0
    n_dec = 0
    for s in np.nonzero(q_lens == 1)[0]:
        kv = int(b.kv_lens[s])
        j = np.arange(max(0, kv - window) if window > 0 else 0, kv)
        slots.append(b.block_table[s][j // b.block_size].astype(np.int64) * b.block_size
                     + j % b.block_size)
        logical += j.size
        n_dec += 1
    unique = int(np.unique(np.concatenate(slots)).size) if slots else 0
    qo = n_dec * b.num_q_heads * b.head_dim * 2 * 2
    return unique * row_bytes + qo, logical * row_bytes + qo


def chunk_flops(b: workloads.Batch, window: int = 0):
    """Algorithmic FLOPs of the chunk pass: 4 * D * Hq per unmasked (query, key) pair."""
    q_lens = np.diff(b.cu_seqlens_q)
    pairs = 0
    for s in np.nonzero(q_lens > 1)[0]:
        n = int(q_lens[s])
        ctx = int(b.kv_lens[s]) - n
        if window > 0:
            pos = np.arange(ctx, ctx + n) + 1          # keys visible: min(position + 1, W)
            pairs += int(np.minimum(pos, window).sum())
        else:
            pairs += n * ctx + n * (n + 1) // 2
    return 4.0 * b.head_dim * b.num_q_heads * pairs


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "continuous_batching_paged_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[f"{kernel}:{workload}"]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != source_hash(*rec.get("sources", [])):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock and the throttle reasons seen, over the samples taken between host
        times t0 and t1 (all samples when not given; the whole run if that window caught none,
        which a window shorter than the 100 ms sampling period can)."""
        lines = [l for t, l in self.lines if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if not lines and t0 is not None:
            lines = [l for t, l in self.lines if t >= t0 - 0.15] or [l for _, l in self.lines]
        rows = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                sm, smax, pw, util = float(parts[0]), float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            rows.append((sm, smax, pw, util, parts[4:]))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r[3] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(busy),
                "power_w_max": max(r[2] for r in busy)}


# ----------------------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if (torch.cuda.is_available() and args.impl == "cb") else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def dist_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle timing

class BenchBatch:
    """A named batch for the bench: the seeded layout (lengths, block tables) of
    workloads.make_layout, with its values drawn N(0, 1) in bf16 by torch's generator on
    `device` (K scaled by the layout's k_scale); pages outside the batch's tables hold values
    too.  The oracle's sample copies the values it needs back from the device."""

    def __init__(self, lay: workloads.Layout, seed: int, device):
        import torch
        self.lay = lay
        self.device = device
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        T, Hq, Hkv, D = lay.num_tokens, lay.num_q_heads, lay.num_kv_heads, lay.head_dim

        def draw(shape, scale=1.0):
            x = torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
            return x.mul_(scale) if scale != 1.0 else x   # 4 = 2^2: exact in bf16

        self.k_pages = draw((lay.num_pages, lay.block_size, Hkv, D), lay.k_scale)
        self.v_pages = draw((lay.num_pages, lay.block_size, Hkv, D))
        self.q = draw((T, Hq, D))
        self.k_new = draw((T, Hkv, D), lay.k_scale)
        self.v_new = draw((T, Hkv, D))
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
        self.table, self.cu, self.kv = i32(lay.block_table), i32(lay.cu_seqlens_q), i32(lay.kv_lens)
        self.q_h, self.k_new_h, self.v_new_h = (_bits(x) for x in (self.q, self.k_new, self.v_new))

    def pages(self, ids: np.ndarray):
        """bf16 bits of blocks `ids` of both pools, copied from the device."""
        import torch
        idx = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int64)).to(self.device)
        return _bits(self.k_pages.index_select(0, idx)), _bits(self.v_pages.index_select(0, idx))


class HostBenchBatch:
    """The reference arm's batch: the same seeded layout as BenchBatch, with values drawn on
    the host on demand (each block from its own seeded generator), so that the oracle's sample
    costs only the blocks it reads."""

    def __init__(self, lay: workloads.Layout, seed: int):
        self.lay = lay
        self.seed = seed
        rng = np.random.default_rng([seed, 1])
        T, Hq, Hkv, D = lay.num_tokens, lay.num_q_heads, lay.num_kv_heads, lay.head_dim
        self.q_h = workloads.f32_to_bf16_bits(rng.standard_normal((T, Hq, D), dtype=np.float32))
        self.k_new_h = workloads.f32_to_bf16_bits(
            lay.k_scale * rng.standard_normal((T, Hkv, D), dtype=np.float32))
        self.v_new_h = workloads.f32_to_bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32))

    def pages(self, ids: np.ndarray):
        lay = self.lay
        shape = (lay.block_size, lay.num_kv_heads, lay.head_dim)
        k = np.empty((len(ids),) + shape, dtype=np.uint16)
        v = np.empty_like(k)
        for i, blk in enumerate(ids):
            rng = np.random.default_rng([self.seed, 2, int(blk)])
            k[i] = workloads.f32_to_bf16_bits(lay.k_scale * rng.standard_normal(shape, dtype=np.float32))
            v[i] = workloads.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        return k, v


def _bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def sub_batch(bb, seqs, chunk_rows=None) -> workloads.Batch:
    """The listed sequences of the bench batch as a host batch of their own (a chunk keeps its
    prior context and its first chunk_rows queries; only the blocks they reference)."""
    lay = bb.lay
    q_lens = lay.q_lens
    new_q, new_kv, rows = [], [], []
    for s in seqs:
        n = int(q_lens[s])
        ctx = int(lay.kv_lens[s]) - n
        if chunk_rows is not None and n > chunk_rows:
            n = chunk_rows
        c0 = int(lay.cu_seqlens_q[s])
        rows.append(np.arange(c0, c0 + n))
        new_q.append(n)
        new_kv.append(ctx + n)
    rows = np.concatenate(rows)
    cu = np.zeros(len(seqs) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(new_q)
    table = lay.block_table[list(seqs)].copy()
    used = np.unique(table[table >= 0])
    remap = np.full(lay.num_pages, -1, dtype=np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    table = np.where(table >= 0, remap[np.maximum(table, 0)], -1).astype(np.int32)
    kp, vp = bb.pages(used)
    return workloads.Batch(name=lay.name + "-sample", q=bb.q_h[rows], k_new=bb.k_new_h[rows],
                           v_new=bb.v_new_h[rows], k_pages=kp, v_pages=vp, block_table=table,
                           cu_seqlens_q=cu, kv_lens=np.asarray(new_kv, dtype=np.int32),
                           block_size=lay.block_size, scale=lay.scale,
                           num_q_heads=lay.num_q_heads, num_kv_heads=lay.num_kv_heads,
                           head_dim=lay.head_dim)


def oracle_step(sb: workloads.Batch, window: int = 0):
    """Append + attention of the sample in the oracle; returns its output rows [T, Hq, D]."""
    from oracle import paged_attention as opa
    kp, vp = opa.kv_append(sb.k_new, sb.v_new, sb.k_pages, sb.v_pages, sb.block_table,
                           sb.cu_seqlens_q, sb.kv_lens, sb.block_size)
    out, _ = opa.ragged_paged_attention(sb.q, kp, vp, sb.block_table, sb.cu_seqlens_q,
                                        sb.kv_lens, sb.block_size, sb.scale, window=window)
    return out


def sample_rows(lay, seqs, chunk_rows=128):
    """Token indices of the full batch that sub_batch(.., seqs, chunk_rows) keeps, in order."""
    q_lens = lay.q_lens
    rows = []
    for s in seqs:
        c0 = int(lay.cu_seqlens_q[s])
        rows.extend(range(c0, c0 + min(int(q_lens[s]), chunk_rows)))
    return np.asarray(rows, dtype=np.int64)


def parity_of(gpu_rows: np.ndarray, ref: np.ndarray):
    """The bench's own parity line: the CUDA output rows of the oracle's sample against the
    oracle, with the bar the parity tests use (|gpu - ref| <= 2e-2 + 1e-2 |ref|)."""
    gpu = gpu_rows.astype(np.float64)
    err = np.abs(gpu - ref)
    return {"rows_checked": int(ref.shape[0]), "values_checked": int(ref.size),
            "max_abs_err": float(err.max()), "max_rel_err": float((err / np.maximum(np.abs(ref), 1e-3)).max()),
            "within_bar": bool(np.isfinite(gpu).all() and (err <= 2e-2 + 1e-2 * np.abs(ref)).all()),
            "bar": "|gpu - ref| <= 2e-2 + 1e-2 |ref| elementwise"}


def cpu_sample_plan(bb, budget_s: float, window: int = 0):
    """A bounded sample: decode sequences and (for chunks) the first 128 queries of each chunk,
    grown until one oracle pass takes about budget_s."""
    q_lens = bb.lay.q_lens
    dec = [int(s) for s in np.nonzero(q_lens == 1)[0]]
    chunks = [int(s) for s in np.nonzero(q_lens > 1)[0]]
    order = []
    for i in range(max(len(dec), len(chunks))):
        if i < len(chunks):
            order.append(chunks[i])
        if i < len(dec):
            order.append(dec[i])
    n = 1
    while True:
        sb = sub_batch(bb, order[:n], chunk_rows=128)
        t0 = time.perf_counter()
        oracle_step(sb, window)
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= len(order):
            return order[:n], sb, dt
        n = min(len(order), max(n + 1, int(n * min(4.0, budget_s / max(dt, 1e-3)))))


_ONE_THREAD = """
import pickle, sys, time
sys.path.insert(0, sys.argv[1])
import bench
from oracle import paged_attention  # noqa: F401  (imported before the clock starts)
sb, window = pickle.load(sys.stdin.buffer)
t0 = time.perf_counter()
bench.oracle_step(sb, window)
print(time.perf_counter() - t0)
"""


def oracle_seconds_one_thread(sb: workloads.Batch, window: int = 0):
    """The same oracle pass in a child process whose BLAS / OpenMP pools have one thread."""
    import pickle
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", _ONE_THREAD, ROOT], input=pickle.dumps((sb, window)),
                           capture_output=True, env=env, timeout=300)
        return float(r.stdout.decode().strip().splitlines()[-1]) if r.returncode == 0 else None
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        return None


def cpu_baseline(bb: BenchBatch, budget_s: float = 15.0, gpu_out=None, window: int = 0,
                 one_thread: bool = True):
    seqs, sb, _ = cpu_sample_plan(bb, budget_s / 2, window)
    t0 = time.perf_counter()
    ref = oracle_step(sb, window)
    dt = time.perf_counter() - t0
    toks = int(sb.cu_seqlens_q[-1])
    dt1 = oracle_seconds_one_thread(sb, window) if one_thread else None
    parity = None
    if gpu_out is not None:  # the CUDA path's rows of the same sample, as float32 numpy
        parity = parity_of(gpu_out(sample_rows(bb.lay, seqs)), ref)
    return {"value": toks / dt, "unit": "query tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "seconds": dt, "parity_vs_cuda": parity,
            "threads": "numpy's default BLAS / OpenMP pools (one per core)",
            "one_thread": None if dt1 is None else {"value": toks / dt1, "cores": 1,
                                                    "seconds": dt1},
            "sample": f"{len(seqs)} of {bb.lay.num_seqs} sequences of the same batch ({toks} query "
                      f"tokens; chunks cut to their first 128 queries at their own prior context; "
                      f"only their referenced blocks), append + attention in float64 numpy, "
                      f"{dt:.2f} s"}


def run_reference(args, lay: workloads.Layout, seed: int, rank: int, world: int):
    if rank != 0:
        return
    bb = HostBenchBatch(lay, seed)
    total = args.steps + args.warmup
    per_step = max(0.05, min(2.0, 150.0 / max(total, 1)))
    seqs, sb, _ = cpu_sample_plan(bb, per_step, args.window)
    for _ in range(args.warmup):
        oracle_step(sb, args.window)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sb, args.window)
    dt = time.perf_counter() - t0
    toks = int(sb.cu_seqlens_q[-1])
    value = toks * args.steps / dt
    unit = "query tokens/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(lay, args.workload, args),
        "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "value": value, "unit": unit,
                         "sample": f"each step: {len(seqs)} of {lay.num_seqs} sequences "
                                   f"({toks} query tokens; chunks cut to 128 queries)"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(lay: workloads.Layout, name: str, args, overrides=None):
    cfg = WORKLOADS[name] if name in WORKLOADS else None
    desc = workloads.CONFIGS[cfg] if cfg is not None else name
    if overrides:
        desc += " -- with " + ", ".join(f"{k}={v}" for k, v in overrides.items())
    return {"workload": desc, "seqs": lay.num_seqs,
            "query_tokens": lay.num_tokens, "q_heads": lay.num_q_heads,
            "kv_heads": lay.num_kv_heads, "head_dim": lay.head_dim, "block_size": lay.block_size,
            "pages": lay.num_pages,
            "l2": "flushed before every timed step (512 MiB write, then 512 MiB read); KV also exceeds L2",
            "parallelism": f"replicas x{args.gpus}",
            "values": "N(0,1) bf16 from torch's seeded device generator; lengths and block "
                      "tables from the seeded layout",
            **({"window": args.window} if getattr(args, "window", 0) else {})}


# ----------------------------------------------------------------------------- GPU arm

def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def run_blocks(args, local: int):
    """Block-move kernels on a 16384-block pool (bs 32, 8 KV heads, D 128: 64 KB per block and
    pool): copy-on-write copies of 4096 disjoint block pairs inside HBM, and the offload /
    restore of 4096 blocks to pinned host memory, each against its own roofline (the measured
    HBM copy peak; a contiguous cudaMemcpy of the same bytes over the same CPU-GPU link)."""
    import torch
    import continuous_batching_paged_gb300 as cb
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P, bs, H, D, n = 16384, 32, 8, 128, 4096
    kp = torch.randn((P, bs, H, D), device=dev).to(torch.bfloat16)
    vp = torch.randn((P, bs, H, D), device=dev).to(torch.bfloat16)
    g = torch.Generator().manual_seed(1234)
    perm = torch.randperm(P, generator=g)
    src, dst = perm[:n].to(torch.int32).to(dev), perm[n:2 * n].to(torch.int32).to(dev)
    blocks = perm[2 * n:3 * n].to(torch.int32).to(dev)
    hk = torch.empty((n, bs, H, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((n, bs, H, D), dtype=torch.bfloat16).pin_memory()
    block_bytes = bs * H * D * 2
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    dbuf = torch.empty((2 * n, bs, H, D), dtype=torch.bfloat16, device=dev)
    hbuf = torch.empty((2 * n, bs, H, D), dtype=torch.bfloat16).pin_memory()

    def timed(fn, reps):
        e0, e1 = _events(torch, 2)
        tot = 0.0
        for i in range(args.warmup + reps):
            flush.fill_(1.0)
            flush_r.sum()
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            if i >= args.warmup:
                tot += e0.elapsed_time(e1)
        return tot / reps / 1e3  # seconds

    reps = max(3, min(args.steps, 20))
    t_copy = timed(lambda: cb.copy_blocks(kp, vp, src, dst, bs), reps)
    t_off = timed(lambda: cb.kv_offload(kp, vp, blocks, bs, hk, hv), reps)
    t_res = timed(lambda: cb.kv_restore(kp, vp, blocks, bs, hk, hv), reps)
    t_d2h = timed(lambda: hbuf.copy_(dbuf, non_blocking=True), reps)
    t_h2d = timed(lambda: dbuf.copy_(hbuf, non_blocking=True), reps)
    cb.check_device_error()
    pk, pk_kind = peaks()
    moved = 2 * n * block_bytes                      # K and V blocks
    copy_gbs = 2 * moved / t_copy / 1e9              # read + write
    line = {
        "metric": "KV block moves GB/s (copy-on-write copy in HBM; offload / restore over the "
                  "CPU-GPU link)", "mode": "blocks", "n_gpus": 1, "data": "synthetic",
        "config": {"pool_blocks": P, "block_size": bs, "kv_heads": H, "head_dim": D,
                   "blocks_per_call": n, "bytes_per_call_each_way": moved,
                   "l2": "flushed before every timed call (512 MiB write, then 512 MiB read)"},
        "copy_blocks": {"ms": t_copy * 1e3, "gbs": copy_gbs, "peak_gbs": pk["hbm_gbs"],
                        "frac": copy_gbs / pk["hbm_gbs"], "peak_kind": pk_kind + " HBM copy"},
        "kv_offload": {"ms": t_off * 1e3, "gbs": moved / t_off / 1e9,
                       "contiguous_d2h_gbs": moved / t_d2h / 1e9,
                       "frac_of_contiguous": t_d2h / t_off},
        "kv_restore": {"ms": t_res * 1e3, "gbs": moved / t_res / 1e9,
                       "contiguous_h2d_gbs": moved / t_h2d / 1e9,
                       "frac_of_contiguous": t_h2d / t_res},
        "gpu_launches": 3 * reps,
    }
    print(json.dumps(line), flush=True)


def run_serve(args, local: int):
    """A continuous-batching serving loop driven by the native scheduler: 1024 requests
    (prompt lognormal, median 512, sigma 1, capped at 4096; 64-512 new tokens), all queued at
    the start, FIFO (or PrefillFirst) under max_batch_tokens 2048 and 256 requests per step on
    a 64k-block pool (bs 32, 32 query / 8 KV heads, D 128).  Every step: the scheduler builds
    the batch on the host, its metadata goes to the device from pinned buffers, then the
    block copies, the KV append and the attention pass run.  Query/key/value rows come from a
    pre-drawn random buffer (no model).  Reports query tokens per second of the whole loop
    (host scheduling and launches included), the device time per step, and the host time of
    the scheduler per step."""
    import numpy as np
    import torch
    import continuous_batching_paged_gb300 as cb
    from continuous_batching_paged_gb300.runtime import BlockAllocator, Scheduler
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P, bs, Hq, Hkv, D, MB = 65536, 32, 32, 8, 128, 160
    budget, cap = 2048, 256
    rng = np.random.default_rng(2024)
    n_req = 1024
    prompts = np.minimum(np.exp(np.log(512) + rng.standard_normal(n_req)), 4096).astype(int) + 1
    news = rng.integers(64, 513, n_req)
    alloc = BlockAllocator(P, bs, MB)
    sched = Scheduler(alloc, budget, cap, args.policy)
    for i in range(n_req):
        sched.add_request(i, int(prompts[i]), int(news[i]))
    kp = torch.zeros((P, bs, Hkv, D), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros((P, bs, Hkv, D), dtype=torch.bfloat16, device=dev)
    q_all = torch.randn((budget, Hq, D), device=dev).to(torch.bfloat16)
    k_all = torch.randn((budget, Hkv, D), device=dev).to(torch.bfloat16)
    v_all = torch.randn((budget, Hkv, D), device=dev).to(torch.bfloat16)
    out = torch.empty_like(q_all)
    ws = torch.empty(cb.workspace_size(cap, Hq, Hkv, D, budget), dtype=torch.uint8,
                     device=dev)
    nbuf = 3  # pinned metadata ring: the host fills step k+1 while the GPU reads step k
    h_meta = [torch.empty(cap + 1 + cap + cap * MB + 2 * cap, dtype=torch.int32).pin_memory()
              for _ in range(nbuf)]
    d_meta = [torch.empty(cap + 1 + cap + cap * MB + 2 * cap, dtype=torch.int32, device=dev)
              for _ in range(nbuf)]
    done_ev = [None] * nbuf
    stream = torch.cuda.current_stream()
    lib = cb.library()
    scale = 1.0 / float(np.sqrt(D))

    def one_step(k):
        t0 = time.perf_counter()
        st = sched.step()
        t_sched = time.perf_counter() - t0
        S, T = len(st["seq_ids"]), int(st["num_tokens"])
        if S == 0:
            return 0, t_sched
        slot = k % nbuf
        if done_ev[slot] is not None:
            done_ev[slot].synchronize()
        h = h_meta[slot].numpy()
        o = 0
        h[o:o + S + 1] = st["cu_seqlens_q"]; cu_o = o; o += cap + 1
        h[o:o + S] = st["kv_lens"]; kv_o = o; o += cap
        h[o:o + S * MB] = st["block_table"].reshape(-1); tb_o = o; o += cap * MB
        nc = len(st["cow_src"])
        h[o:o + nc] = st["cow_src"]; src_o = o; o += cap
        h[o:o + nc] = st["cow_dst"]; dst_o = o
        d = d_meta[slot]
        d.copy_(h_meta[slot], non_blocking=True)
        cu_d, kv_d = d[cu_o:cu_o + S + 1], d[kv_o:kv_o + S]
        tb_d = d[tb_o:tb_o + S * MB].view(S, MB)
        if nc:
            cb.copy_blocks(kp, vp, d[src_o:src_o + nc], d[dst_o:dst_o + nc], bs)
        cb.kv_append(k_all[:T], v_all[:T], kp, vp, tb_d, cu_d, kv_d, bs)
        cb.ragged_paged_attention(q_all[:T], kp, vp, tb_d, cu_d, kv_d, bs, scale,
                                  out=out[:T], workspace=ws)
        ev = torch.cuda.Event()
        ev.record(stream)
        done_ev[slot] = ev
        return T, t_sched

    warm = max(3, args.warmup)
    for k in range(warm):
        one_step(k)
    torch.cuda.synchronize()
    e0, e1 = _events(torch, 2)
    tokens, steps, t_sched = 0, 0, 0.0
    limit = max(args.steps, 50)
    wall0 = time.perf_counter()
    e0.record()
    while steps < limit and sched.num_active():
        T, ts = one_step(warm + steps)
        tokens += T
        t_sched += ts
        steps += 1
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    cb.check_device_error()
    dev_ms = e0.elapsed_time(e1)
    line = {
        "metric": "continuous-batching loop query tokens/s (native scheduler + append + attention)",
        "mode": "serve", "policy": args.policy, "n_gpus": 1, "data": "synthetic",
        "value": tokens / wall, "unit": "query tokens/s", "steps": steps,
        "tokens": tokens, "wall_ms_per_step": 1e3 * wall / steps,
        "device_ms_per_step": dev_ms / steps,
        "sched_us_per_step": 1e6 * t_sched / steps,
        "config": {"requests": n_req, "prompt": "lognormal median 512 sigma 1 cap 4096",
                   "new_tokens": "U[64, 512]", "max_batch_tokens": budget,
                   "max_requests_per_batch": cap, "pool_blocks": P, "block_size": bs,
                   "q_heads": Hq, "kv_heads": Hkv, "head_dim": D},
        "gpu_launches": "3 per step (append, plan, attention; block copy when needed)",
    }
    print(json.dumps(line), flush=True)


def run_graphs(args, local: int):
    """Latency of one step (append + attention, from the call to its completion on the GPU)
    issued eagerly through the Python API vs replayed from a captured CUDA graph, for decode
    batches of 1, 8 and 64 sequences (kv_len 1024) and the 2048-token mixed batch."""
    import torch
    import continuous_batching_paged_gb300 as cb
    from continuous_batching_paged_gb300.graphs import GraphedStep
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shapes = [("decode x1", [1], [1024]), ("decode x8", [1] * 8, [1024] * 8),
              ("decode x64", [1] * 64, [1024] * 64), ("mixed 2048", None, None)]
    rows = []
    for name, ql, kl in shapes:
        b = (workloads.make_config(3) if ql is None else
             workloads.build_batch(ql, kl, 32, 8, 128, 32, seed=77, name=name))
        t16 = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)
        t32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev)
        q, kn, vn = t16(b.q), t16(b.k_new), t16(b.v_new)
        kp, vp = t16(b.k_pages), t16(b.v_pages)
        tab, cu, kv = t32(b.block_table), t32(b.cu_seqlens_q), t32(b.kv_lens)
        out = torch.empty_like(q)
        ws = torch.empty(cb.workspace_size(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                           b.num_tokens),
                         dtype=torch.uint8, device=dev)

        def eager():
            cb.kv_append(kn, vn, kp, vp, tab, cu, kv, b.block_size)
            cb.ragged_paged_attention(q, kp, vp, tab, cu, kv, b.block_size, b.scale, out=out,
                                      workspace=ws)

        g = GraphedStep(kp, vp, b.block_size, b.scale, b.num_q_heads, b.max_blocks)
        g.run(q, kn, vn, tab, cu, kv)                 # capture, inputs into the graph buffers
        bucket = g.buffers(b.num_seqs, b.num_tokens)

        def graph():
            g.run(q, kn, vn, tab, cu, kv)

        def replay():
            g.replay(bucket)

        res = {}
        for label, fn in (("eager", eager), ("graph", graph), ("replay", replay)):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(max(20, min(args.steps, 200))):
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
            res[label] = 1e6 * statistics.median(ts)
        cb.check_device_error()
        rows.append({"batch": name, "seqs": b.num_seqs, "tokens": b.num_tokens,
                     "eager_us": res["eager"], "graph_with_input_copies_us": res["graph"],
                     "replay_inputs_in_place_us": res["replay"],
                     "speedup_in_place": res["eager"] / res["replay"]})
    print(json.dumps({"metric": "step latency (append + attention, call to completion), eager "
                                "Python API vs CUDA-graph replay", "mode": "graphs", "n_gpus": 1,
                      "data": "synthetic", "unit": "us (median)", "rows": rows,
                      "note": "graph_with_input_copies copies the step's inputs into the graph's "
                              "static buffers first; replay_inputs_in_place is for a producer "
                              "that writes them there (GraphedStep.buffers)"}), flush=True)


# Further batches measured in the same run, after the headline batch: the other named
# workloads, then shapes around the decode-only batch (its lengths with another GQA group
# size, head dim or block size).  (key, named workload, shape overrides, oracle budget in
# seconds, one-thread oracle figure too)
SUB_WORKLOADS = [
    ("decode", 2, {}, 3.0, True),
    ("prefill", 4, {}, 3.0, False),
    ("longtail", 5, {}, 3.0, False),
    ("tiny", 1, {}, 1.0, True),
    ("decode_gqa16", 2, {"num_q_heads": 128}, 1.0, False),
    ("decode_d64", 2, {"head_dim": 64}, 1.0, False),
    ("decode_bs16", 2, {"block_size": 16, "num_pages": 32768}, 1.0, False),
    ("decode_bs4", 2, {"block_size": 4, "num_pages": 131072}, 1.0, False),
]


def measure(args, cb, torch, dev, bb: BenchBatch, world: int, sampler, with_e2e: bool,
            cpu_budget: float, one_thread: bool, rank: int, name: str, overrides=None):
    """Time one batch's step (append + attention) and return its part of the JSON line."""
    lay = bb.lay
    q, kn, vn, kp, vp = bb.q, bb.k_new, bb.v_new, bb.k_pages, bb.v_pages
    table, cu, kvl = bb.table, bb.cu, bb.kv
    out = torch.empty_like(q)
    ws = torch.empty(cb.workspace_size(lay.num_seqs, lay.num_q_heads, lay.num_kv_heads,
                                       lay.head_dim, lay.num_tokens), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write 512 MiB (evicts everything the last step left in the 129 MB L2), then read
        # another 512 MiB, so the step starts on an L2 holding neither its inputs nor dirty
        # lines whose write-back would be charged to the step's own DRAM traffic.
        flush.fill_(1.0)
        flush_r.sum()

    # ev_start / ev_end bracket the step on the launching stream; the library records its five
    # phase events around the planner and the attention launch (cb_options).
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ph = [torch.cuda.Event(enable_timing=True) for _ in range(cb.NUM_PHASE_EVENTS)]
    for e in [ev_start, ev_end] + ph:
        e.record()

    def step(record):
        kw = dict(out=out, workspace=ws, decode_ctas=args.decode_ctas,
                  phase_events=ph if record else None, serial=args.serial, window=args.window)
        if args.separate:
            cb.kv_append(kn, vn, kp, vp, table, cu, kvl, lay.block_size)
            cb.ragged_paged_attention(q, kp, vp, table, cu, kvl, lay.block_size, lay.scale, **kw)
        else:
            cb.append_attention(q, kn, vn, kp, vp, table, cu, kvl, lay.block_size, lay.scale, **kw)

    # correctness guard before timing: the error word must be clear after one step
    step(False)
    cb.check_device_error()
    for _ in range(args.warmup):
        flush_l2()
        step(False)
    torch.cuda.synchronize()

    # Timed region: K steps, each bracketed by ev_start / ev_end on the launching stream; no
    # phase events inside (an event between two kernels costs the step a few microseconds).
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms = 0.0
    per_step = []
    for _ in range(args.steps):
        flush_l2()
        ev_start.record()
        step(False)
        ev_end.record()
        ev_end.synchronize()
        per_step.append(ev_start.elapsed_time(ev_end))
        step_ms += per_step[-1]
    torch.cuda.synchronize()
    barrier(world)
    wall1 = time.perf_counter()
    cb.check_device_error()
    ms = dist_max(step_ms / args.steps, world, dev)

    # Kernel spans (roofline inputs): the same steps again with the library's phase events.
    # In the default (one attention launch) mode the decode and chunk passes share a launch:
    # the events time that launch, and the passes' own spans inside it come from the device
    # time stamps the kernel leaves in the workspace (cb_pass_timestamps).
    if args.serial and args.separate:
        spans = {"append": (ev_start, ph[0]), "plan": (ph[0], ph[1]), "decode": (ph[1], ph[2]),
                 "chunk": (ph[3], ph[4])}
    elif args.serial:
        spans = {"append+plan": (ev_start, ph[1]), "decode": (ph[1], ph[2]),
                 "chunk": (ph[3], ph[4])}
    elif args.separate:
        spans = {"append": (ev_start, ph[0]), "plan": (ph[0], ph[1]), "attention": (ph[1], ph[2])}
    else:
        spans = {"append+plan": (ev_start, ph[1]), "attention": (ph[1], ph[2])}
    acc = {n: 0.0 for n in spans}
    role = {"decode": 0.0, "chunk": 0.0}
    n_span = max(1, min(args.steps, 30))
    for _ in range(n_span):
        flush_l2()
        ev_start.record()
        step(True)
        ev_end.record()
        ev_end.synchronize()
        for n, (e0_, e1_) in spans.items():
            acc[n] += e0_.elapsed_time(e1_)
        ts = cb.pass_timestamps(ws)
        role["decode"] += (ts[1] - ts[0]) * 1e-6
        role["chunk"] += (ts[3] - ts[2]) * 1e-6
    cb.check_device_error()
    per_kernel = {n: dist_max(acc[n] / n_span, world, dev) for n in spans}
    role_ms = {n: dist_max(v / n_span, world, dev) for n, v in role.items()}

    e2e = None
    if with_e2e:
        e2e = measure_e2e(args, cb, torch, dev, bb, ws, out, flush_l2, world)

    pk, pk_kind = peaks()
    dec_bytes, dec_logical = decode_kv_bytes(lay, args.window)
    flops = chunk_flops(lay, args.window)
    # Pass spans: with both passes in one launch, from the kernel's device time stamps; in
    # serial mode (two launches), from the events around each launch.
    dec_ms = per_kernel["decode"] if args.serial else role_ms["decode"]
    chunk_ms = per_kernel["chunk"] if args.serial else role_ms["chunk"]
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9 if dec_ms > 0 and dec_bytes else None
    chunk_tf = flops / (chunk_ms * 1e-3) / 1e12 if chunk_ms > 0 and flops else None
    # The roofline is taken on the attention kernel (one launch runs both passes; its span from
    # the events around it), against the bound of the pass with the larger ideal time (work /
    # peak).  In serial mode each pass is its own launch and is measured alone.
    dec_ideal = dec_bytes / (pk["hbm_gbs"] * 1e9) if dec_bytes else 0.0
    chunk_ideal = flops / (pk["bf16_tflops"] * 1e12) if flops else 0.0
    hbm_bound = dec_ideal >= chunk_ideal and dec_bytes > 0
    if args.serial:
        attn_ms = dec_ms if hbm_bound else chunk_ms
    else:
        attn_ms = per_kernel["attention"]
    traffic = recorded_traffic("attention_kernel", name) if not overrides else None
    if hbm_bound:
        ach = dec_bytes / (attn_ms * 1e-3) / 1e9
        roof = {"kernel": "attention_kernel", "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "traffic": traffic,
                "algorithmic_bytes_per_launch": dec_bytes, "launch_ms": attn_ms,
                "peak_kind": pk_kind, "frac_of_nominal_8000": ach / NOMINAL_HBM_GBS}
    else:
        tpk = pk["bf16_tflops"]
        ach = flops / (attn_ms * 1e-3) / 1e12
        roof = {"kernel": "attention_kernel", "bound": "tensor", "achieved": ach, "peak": tpk,
                "unit": "TFLOP/s", "frac": ach / tpk, "traffic": traffic,
                "algorithmic_flops_per_launch": flops, "launch_ms": attn_ms,
                "peak_kind": pk_kind + " burst bf16"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(
            bb, budget_s=cpu_budget, window=args.window, one_thread=one_thread,
            gpu_out=lambda rows: out[torch.from_numpy(rows).to(dev)].float().cpu().numpy())

    res = {
        "value": world * lay.num_tokens / (ms / 1000.0), "unit": "query tokens/s",
        "ms_per_step": ms,
        "step_ms_stats": {"median": statistics.median(per_step), "min": min(per_step),
                          "max": max(per_step)},
        "config": workload_config(lay, name, args, overrides),
        "roofline": roof,
        "decode": {"kv_bytes_unique": dec_bytes, "kv_bytes_logical": dec_logical,
                   "span_ms": dec_ms, "gbs": dec_gbs,
                   "frac_of_measured": (dec_gbs / pk["hbm_gbs"]) if dec_gbs else None,
                   "frac_of_nominal_8000": (dec_gbs / NOMINAL_HBM_GBS) if dec_gbs else None},
        "chunk": {"flops": flops, "span_ms": chunk_ms, "tflops": chunk_tf,
                  "span_note": None if args.serial else
                  "decode and chunk spans: first start to last end of each pass's CTAs with work "
                  "(device %globaltimer stamps, cb_pass_timestamps); the chunk pass runs on the "
                  "SMs the decode pass leaves free",
                  "frac_of_burst": (chunk_tf / pk["bf16_tflops"]) if chunk_tf else None,
                  "frac_of_sustained": (chunk_tf / pk["bf16_tflops_sustained"]) if chunk_tf else None},
        "kernel_ms": per_kernel,
        "clocks": sampler.summary(wall0, wall1),
        "cpu_baseline": cpu,
        "wall_s_timed": wall1 - wall0,
    }
    if e2e is not None:
        res["e2e"] = e2e
    return res


def measure_e2e(args, cb, torch, dev, bb: BenchBatch, ws, out, flush_l2, world):
    """The step through the public API with inputs from pinned host memory, output back."""
    lay = bb.lay
    q, kn, vn, kp, vp = bb.q, bb.k_new, bb.v_new, bb.k_pages, bb.v_pages
    table, cu, kvl = bb.table, bb.cu, bb.kv
    h_q = torch.from_numpy(bb.q_h.view(np.int16)).pin_memory()
    h_k = torch.from_numpy(bb.k_new_h.view(np.int16)).pin_memory()
    h_v = torch.from_numpy(bb.v_new_h.view(np.int16)).pin_memory()
    h_tab = torch.from_numpy(lay.block_table).pin_memory()
    h_cu = torch.from_numpy(lay.cu_seqlens_q).pin_memory()
    h_kv = torch.from_numpy(lay.kv_lens).pin_memory()
    h_out = torch.empty(tuple(q.shape), dtype=torch.int16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_tab, h_cu, h_kv))
    d2h = h_out.numel() * h_out.element_size()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def run(bq, bk, bv, btab, bcu, bkv, bo):
        kw = dict(out=bo, workspace=ws, decode_ctas=args.decode_ctas, serial=args.serial,
                  window=args.window)
        if args.separate:
            cb.kv_append(bk, bv, kp, vp, btab, bcu, bkv, lay.block_size)
            cb.ragged_paged_attention(bq, kp, vp, btab, bcu, bkv, lay.block_size, lay.scale, **kw)
        else:
            cb.append_attention(bq, bk, bv, kp, vp, btab, bcu, bkv, lay.block_size, lay.scale, **kw)

    def e2e_step():
        q.view(torch.int16).copy_(h_q, non_blocking=True)
        kn.view(torch.int16).copy_(h_k, non_blocking=True)
        vn.view(torch.int16).copy_(h_v, non_blocking=True)
        table.copy_(h_tab, non_blocking=True)
        cu.copy_(h_cu, non_blocking=True)
        kvl.copy_(h_kv, non_blocking=True)
        run(q, kn, vn, table, cu, kvl, out)
        h_out.copy_(out.view(torch.int16), non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for _ in range(args.steps):
        flush_l2()
        e0.record()
        e2e_step()
        e1.record()
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_serial_ms = dist_max(e2e_ms / args.steps, world, dev)
    cb.check_device_error()

    # e2e as a serving loop runs it: double-buffered inputs and outputs, the host->device copy
    # of step i+1 and the device->host read of step i-1 on their own streams, overlapping the
    # kernels of step i.  Every step still copies all its inputs in and its output out.
    def dev_set():
        return [torch.empty_like(x) for x in (q, kn, vn, table, cu, kvl, out)]
    bufs = [dev_set(), dev_set()]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp = torch.cuda.current_stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    for ev in h2d_done + comp_done + d2h_done:
        ev.record(comp)

    def piped_step(i):
        j = i & 1
        bq, bk, bv, btab, bcu, bkv, bo = bufs[j]
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[j])          # buffer j's previous step has been computed
            bq.view(torch.int16).copy_(h_q, non_blocking=True)
            bk.view(torch.int16).copy_(h_k, non_blocking=True)
            bv.view(torch.int16).copy_(h_v, non_blocking=True)
            btab.copy_(h_tab, non_blocking=True)
            bcu.copy_(h_cu, non_blocking=True)
            bkv.copy_(h_kv, non_blocking=True)
            h2d_done[j].record(s_in)
        comp.wait_event(h2d_done[j])
        comp.wait_event(d2h_done[j])               # out buffer j has been read back
        run(bq, bk, bv, btab, bcu, bkv, bo)
        comp_done[j].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            h_outs[j].copy_(bo.view(torch.int16), non_blocking=True)
            d2h_done[j].record(s_out)

    for i in range(max(3, args.warmup)):
        piped_step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.steps):
        piped_step(i)
    torch.cuda.synchronize()
    e2e_ms = dist_max(1e3 * (time.perf_counter() - t0) / args.steps, world, dev)
    cb.check_device_error()
    return {"value": world * lay.num_tokens / (e2e_ms / 1000.0), "unit": "query tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "how": "wall clock over K steps; each step copies its inputs from pinned host "
                   "memory and reads its output back, overlapped with the neighbouring "
                   "steps' kernels (double buffers, copy streams)",
            "serial_ms_per_step": e2e_serial_ms,
            "serial_value": world * lay.num_tokens / (e2e_serial_ms / 1000.0)}


def main():
    args = parse_args()
    if args.mode != "path":
        world, rank, local = dist_setup(args)
        if rank == 0:
            {"blocks": run_blocks, "serve": run_serve, "graphs": run_graphs}[args.mode](args, local)
        return
    world, rank, local = dist_setup(args)
    cfg = WORKLOADS[args.workload]
    seed = 1000 + cfg + 7919 * rank
    lay = workloads.make_layout(cfg, seed=seed)
    if args.impl == "reference":
        run_reference(args, lay, seed, rank, world)
        return

    import torch
    import continuous_batching_paged_gb300 as cb
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the CUDA path has no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cb.library()

    sampler = ClockSampler(local)
    sampler.start()
    bb = BenchBatch(lay, seed, dev)
    # Let the clock sampler see the GPU under load before the first timed region.
    soak_ws = torch.empty(cb.workspace_size(lay.num_seqs, lay.num_q_heads, lay.num_kv_heads,
                                            lay.head_dim, lay.num_tokens), dtype=torch.uint8,
                          device=dev)
    t_start = time.perf_counter()
    n = 0
    while time.perf_counter() - t_start < 2.0:
        cb.append_attention(bb.q, bb.k_new, bb.v_new, bb.k_pages, bb.v_pages, bb.table, bb.cu,
                            bb.kv, lay.block_size, lay.scale, workspace=soak_ws,
                            window=args.window)
        n += 1
        if n % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    del soak_ws

    head = measure(args, cb, torch, dev, bb, world, sampler, with_e2e=True, cpu_budget=15.0,
                   one_thread=True, rank=rank, name=args.workload)
    del bb
    torch.cuda.empty_cache()

    subs = {}
    if not args.only:
        for key, n_cfg, over, budget, one_thr in SUB_WORKLOADS:
            if key == args.workload:
                continue
            s_seed = 1000 + n_cfg + 7919 * rank
            sub_lay = workloads.make_layout(n_cfg, seed=s_seed, **over)
            sbb = BenchBatch(sub_lay, s_seed, dev)
            base = [k for k, v in WORKLOADS.items() if v == n_cfg][0]
            subs[key] = measure(args, cb, torch, dev, sbb, world, sampler, with_e2e=False,
                                cpu_budget=budget, one_thread=one_thr, rank=rank, name=base,
                                overrides=over or None)
            del sbb
            torch.cuda.empty_cache()
    sampler.stop()

    line = {
        "metric": METRIC, "value": head["value"], "unit": "query tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "step_ms_stats": head["step_ms_stats"],
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": head["config"],
        "e2e": head["e2e"],
        # per step: append + plan (one launch) and attention (decode, merge, chunk in one
        # launch); --separate: append, plan, attention; --serial: one more (the passes apart)
        "gpu_launches": (2 + int(args.separate) + int(args.serial)) * args.steps,
        "append_attention": "two calls" if args.separate else "cb_append_attention",
        "concurrent_decode_chunk": not args.serial,
        "roofline": head["roofline"],
        "decode": head["decode"],
        "chunk": head["chunk"],
        "kernel_ms": head["kernel_ms"],
        "clocks": head["clocks"],
        "cpu_baseline": head["cpu_baseline"],
        "wall_s_timed": head["wall_s_timed"],
        "workloads": subs,
        "clocks_whole_run": sampler.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
