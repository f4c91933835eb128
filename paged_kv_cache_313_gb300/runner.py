"""One step of the hot path on the device: slot mapping and KV write for every
new token, then decode for the decode sequences and causal chunked prefill for
the prefill chunks — four library calls on one stream.

``DeviceStep`` owns the device copies of a :class:`Workload` and the output
and workspace buffers, so that repeated steps allocate nothing.
"""
from __future__ import annotations

import torch

from . import pa
from .workloads import Workload


class DeviceStep:
    def __init__(self, w: Workload, device: str | torch.device = "cuda", with_error_count: bool = True):
        dev = torch.device(device)
        self.w = w
        self.device = dev
        up = lambda t: t.to(dev).contiguous()  # noqa: E731
        self.k_cache = up(w.k_cache)
        self.v_cache = up(w.v_cache)
        self.block_tables = up(w.block_tables)
        self.context_lens = up(w.context_lens)
        self.seq_idx = up(w.seq_idx)
        self.pos = up(w.pos)
        self.k_new = up(w.k_new)
        self.v_new = up(w.v_new)
        self.q_decode = up(w.q_decode)
        self.cu_q_lens = up(w.cu_q_lens)
        self.q_start_pos = up(w.q_start_pos)
        self.seq_of_chunk = up(w.seq_of_chunk)
        self.q_prefill = up(w.q_prefill)
        self.slots = torch.empty(w.seq_idx.numel(), dtype=torch.int64, device=dev)
        self.out_decode = torch.empty_like(self.q_decode)
        self.out_prefill = torch.empty_like(self.q_prefill)
        self.error_count = torch.zeros(1, dtype=torch.int32, device=dev) if with_error_count else None
        self.max_context_len = w.max_decode_context
        nd = w.num_decode
        self.workspace = (pa.new_decode_workspace(nd, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                                  self.max_context_len, device=dev) if nd else None)
        n = pa.pa_prefill_workspace_size(w.num_chunks, w.max_q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                         w.block_size) if w.num_chunks else 0
        self.prefill_workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=dev) if n else None

    # individual stages --------------------------------------------------
    def slot_mapping(self, stream=None):
        w = self.w
        return pa.pa_slot_mapping(self.block_tables, self.seq_idx, self.pos, w.block_size, w.num_blocks,
                                  slot_mapping=self.slots, error_count=self.error_count, stream=stream)

    def write_kv(self, stream=None):
        pa.pa_write_kv(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slots,
                       error_count=self.error_count, stream=stream)

    def decode(self, stream=None):
        w = self.w
        if not w.num_decode:
            return self.out_decode
        nd = w.num_decode
        return pa.pa_decode(self.q_decode, self.k_cache, self.v_cache, self.block_tables[:nd],
                            self.context_lens[:nd], self.max_context_len, w.scale, self.workspace,
                            out=self.out_decode, error_count=self.error_count, stream=stream)

    def prefill(self, stream=None):
        w = self.w
        if not w.num_chunks:
            return self.out_prefill
        return pa.pa_prefill_chunk(self.q_prefill, self.cu_q_lens, self.q_start_pos, self.seq_of_chunk,
                                   w.max_q_len, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                                   w.scale, workspace=self.prefill_workspace, out=self.out_prefill,
                                   error_count=self.error_count, stream=stream)

    def run(self, stream=None):
        """The whole step: write this step's K/V, then attend."""
        self.slot_mapping(stream)
        self.write_kv(stream)
        self.decode(stream)
        self.prefill(stream)
        return self.out_decode, self.out_prefill

    def capture(self) -> "torch.cuda.CUDAGraph":
        """Record one whole step (the four library calls) as a CUDA graph, so a
        serving loop replays it with one launch.  Call after at least one eager
        step (first calls configure the kernels)."""
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream(self.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self):
        """Replay the captured step on the current stream."""
        self.graph.replay()
        return self.out_decode, self.out_prefill

    def errors(self) -> int:
        return int(self.error_count.item()) if self.error_count is not None else 0
