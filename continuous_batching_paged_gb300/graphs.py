"""The KV append + attention pass of one step captured in CUDA graphs, one graph per padded
batch shape, replayed for every later batch whose padded shape matches.

transformers "Continuous batching architecture", section "CUDA graphs": recording the step's
GPU work once and replaying it removes the per-step CPU dispatch; because batch shapes change
every step, shapes are padded to multiples of an interval and the recorded graphs are kept in
a cache (LRU, bounded).  Here only the shapes that size buffers are padded: the number of
sequences (to a multiple of `seq_interval`, with empty sequences: q_len 0, kv_len 0) and the
number of query tokens (to a multiple of `token_interval`, with padding rows past
cu_seqlens_q[S] that the library neither reads nor writes).  KV lengths need no padding: the
library plans every pass on the device from kv_lens, so one graph serves any lengths.

    g = GraphedStep(k_pages, v_pages, block_size, scale, num_q_heads, max_blocks_per_seq)
    out = g.run(q, k_new, v_new, block_table, cu_seqlens_q, kv_lens)   # view of a graph buffer
"""
from __future__ import annotations

from collections import OrderedDict

from . import append_attention, workspace_size


def _round_up(x: int, m: int) -> int:
    return max(m, -(-x // m) * m)


class _Bucket:
    def __init__(self, owner: "GraphedStep", S: int, T: int):
        import torch
        o = owner
        dev = o.k_pages.device
        self.S, self.T = S, T
        self.q = torch.zeros((T, o.Hq, o.D), dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros((T, o.Hkv, o.D), dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros((T, o.Hkv, o.D), dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros((T, o.Hq, o.D), dtype=torch.bfloat16, device=dev)
        self.cu = torch.zeros(S + 1, dtype=torch.int32, device=dev)
        self.kv = torch.zeros(S, dtype=torch.int32, device=dev)
        self.table = torch.full((S, o.MB), -1, dtype=torch.int32, device=dev)
        self.ws = torch.empty(workspace_size(S, o.Hq, o.Hkv, o.D, T),
                              dtype=torch.uint8, device=dev)

        def body():
            append_attention(self.q, self.k, self.v, o.k_pages, o.v_pages, self.table, self.cu,
                             self.kv, o.bs, o.scale, out=self.out, workspace=self.ws)

        # One eager pass on a side stream (all sequences empty: nothing is read or written)
        # initialises the library on this device before the capture, then the capture.
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            body()
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            body()


class GraphedStep:
    """Append + attention through cached CUDA graphs for padded (sequences, tokens) shapes."""

    def __init__(self, k_pages, v_pages, block_size: int, scale: float, num_q_heads: int,
                 max_blocks_per_seq: int, seq_interval: int = 16, token_interval: int = 64,
                 max_graphs: int = 32):
        self.k_pages, self.v_pages = k_pages, v_pages
        self.bs = int(block_size)
        self.scale = float(scale)
        self.Hq = int(num_q_heads)
        self.Hkv, self.D = int(k_pages.shape[2]), int(k_pages.shape[3])
        self.MB = int(max_blocks_per_seq)
        self.seq_interval, self.token_interval = int(seq_interval), int(token_interval)
        self.max_graphs = int(max_graphs)
        self.cache: OrderedDict[tuple[int, int], _Bucket] = OrderedDict()
        self.captures = 0

    def bucket_of(self, S: int, T: int) -> tuple[int, int]:
        return _round_up(S, self.seq_interval), _round_up(T, self.token_interval)

    def buffers(self, S: int, T: int) -> "_Bucket":
        """The static buffers of the graph for S sequences and T tokens (captured on first use).
        A caller that produces its inputs in place writes q/k/v rows [:T] and the metadata
        cu[:S+1], kv[:S], table[:S] (padding: cu[S+1:] = cu[S], kv[S:] = 0), then calls
        replay(); nothing is copied then."""
        key = self.bucket_of(S, T)
        b = self.cache.get(key)
        if b is None:
            b = _Bucket(self, *key)
            self.captures += 1
            self.cache[key] = b
            if len(self.cache) > self.max_graphs:
                self.cache.popitem(last=False)
        self.cache.move_to_end(key)
        return b

    @staticmethod
    def replay(b: "_Bucket") -> None:
        b.graph.replay()

    def run(self, q, k_new, v_new, block_table, cu_seqlens_q, kv_lens):
        """Copy this step's inputs into the bucket's buffers and replay its graph; returns the
        output rows [T, Hq, D] (a view that the next run of the same bucket overwrites)."""
        S, T = int(kv_lens.numel()), int(q.shape[0])
        b = self.buffers(S, T)
        key = (b.S, b.T)
        b.q[:T].copy_(q)
        b.k[:T].copy_(k_new)
        b.v[:T].copy_(v_new)
        b.cu[:S + 1].copy_(cu_seqlens_q)
        if key[0] > S:
            b.cu[S + 1:].copy_(cu_seqlens_q[S:S + 1].expand(key[0] - S))  # empty sequences
            b.kv[S:].zero_()
        b.kv[:S].copy_(kv_lens)
        b.table[:S, :block_table.shape[1]].copy_(block_table)
        b.graph.replay()
        return b.out[:T]
