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


# Per-step inputs, in the order they sit in the packed input buffer, and outputs.
STEP_INPUTS = ("q_decode", "k_new", "v_new", "block_tables", "context_lens", "seq_idx", "pos", "q_prefill",
               "cu_q_lens", "q_start_pos", "seq_of_chunk", "group_offsets", "prefix_lens")
STEP_OUTPUTS = ("out_decode", "out_prefill")
_ALIGN = 256


def _packed(tensors, device):
    """One uint8 buffer holding every tensor at a 256-byte aligned offset, and
    views of it with each tensor's dtype and shape."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // _ALIGN) * _ALIGN
    buf = torch.empty(max(total, _ALIGN), dtype=torch.uint8, device=device)
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def _packed_views(buf, like):
    """Views of an existing packed buffer laid out like `_packed` lays out `like`."""
    offs, total = [], 0
    for t in like:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // _ALIGN) * _ALIGN
    return buf, [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, like)]


class DeviceStep:
    def __init__(self, w: Workload, device: str | torch.device = "cuda", with_error_count: bool = True,
                 cascade: bool = True, fused_decode_write: bool = True):
        dev = torch.device(device)
        self.w = w
        self.device = dev
        up = lambda t: t.to(dev).contiguous()  # noqa: E731
        self.k_cache = up(w.k_cache)
        self.v_cache = up(w.v_cache)
        # The per-step inputs live in one device buffer (and the outputs in
        # another), so that a serving loop moves a step's inputs in with one
        # host-to-device copy and its outputs out with one copy back.
        host_in = [getattr(w, name).contiguous() for name in STEP_INPUTS]
        self.inbuf, views = _packed(host_in, dev)
        for name, v, t in zip(STEP_INPUTS, views, host_in):
            v.copy_(t)
            setattr(self, name, v)
        self.outbuf, views = _packed([w.q_decode, w.q_prefill], dev)
        for name, v in zip(STEP_OUTPUTS, views):
            setattr(self, name, v)
        self.slots = torch.empty(w.seq_idx.numel(), dtype=torch.int64, device=dev)
        self.error_count = torch.zeros(1, dtype=torch.int32, device=dev) if with_error_count else None
        self.max_context_len = w.max_decode_context
        nd = w.num_decode
        self.workspace = (pa.new_decode_workspace(nd, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                                  self.max_context_len, device=dev) if nd else None)
        # cascade decode when decode sequences share prefixes (and the shapes allow it)
        if w.kv_fp8 and w.num_chunks:
            raise ValueError("e4m3 pools are read by decode only; prefill chunks need bf16 or fp32 pools")
        self.use_cascade = bool(cascade and nd and not w.kv_fp8 and int(w.prefix_lens.max()) > 0
                                and w.dtype == torch.bfloat16
                                and w.head_dim == 128 and w.num_q_heads // w.num_kv_heads in (1, 2, 4, 8)
                                and w.block_size in (8, 16, 32, 64))
        self.cascade_workspace = (pa.new_cascade_workspace(nd, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                           w.block_size, self.max_context_len, device=dev)
                                  if self.use_cascade else None)
        # decode tokens written by the decode kernel itself (pa_decode_write, pa_decode_write_fp8) when the step's first nd new
        # tokens are the decode sequences' newest ones and the shapes are the tensor-core decode kernel's
        G = w.num_q_heads // w.num_kv_heads
        newest = bool(nd) and torch.equal(w.seq_idx[:nd], torch.arange(nd, dtype=w.seq_idx.dtype)) and \
            torch.equal(w.pos[:nd], w.context_lens[:nd].to(w.pos.dtype) - 1)
        dims = (128,) if w.kv_fp8 else (64, 128)  # e4m3 pools: the decode kernel takes head_dim 128
        self.fused_decode_write = bool(fused_decode_write and newest and not self.use_cascade
                                       and w.dtype == torch.bfloat16 and w.head_dim in dims and G <= 8
                                       and w.block_size in (8, 16, 32, 64))
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

    def write_kv_paged(self, stream=None):
        """Slot mapping and K/V write in one launch (the slots are still recorded)."""
        if self.w.kv_fp8:
            pa.pa_write_kv_paged_fp8(self.k_new, self.v_new, self.k_cache, self.v_cache, self.block_tables,
                                     self.seq_idx, self.pos, self.w.k_scale, self.w.v_scale, slot_mapping=self.slots,
                                     error_count=self.error_count, stream=stream)
            return
        pa.pa_write_kv_paged(self.k_new, self.v_new, self.k_cache, self.v_cache, self.block_tables, self.seq_idx,
                             self.pos, slot_mapping=self.slots, error_count=self.error_count, stream=stream)

    def decode(self, stream=None):
        w = self.w
        if not w.num_decode:
            return self.out_decode
        nd = w.num_decode
        if w.kv_fp8:
            return pa.pa_decode_fp8(self.q_decode, self.k_cache, self.v_cache, self.block_tables[:nd],
                                    self.context_lens[:nd], self.max_context_len, w.scale, w.k_scale, w.v_scale,
                                    self.workspace, out=self.out_decode, error_count=self.error_count,
                                    stream=stream)
        if self.use_cascade:
            return pa.pa_decode_cascade(self.q_decode, self.k_cache, self.v_cache, self.block_tables[:nd],
                                        self.context_lens[:nd], self.max_context_len, self.group_offsets,
                                        w.max_group_size, self.prefix_lens, w.scale, self.cascade_workspace,
                                        out=self.out_decode, error_count=self.error_count, stream=stream)
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

    def write_stage(self, stream=None):
        """The step's KV writes that are not done by the decode kernel itself."""
        if not self.fused_decode_write:
            self.write_kv_paged(stream)
            return
        nd = self.w.num_decode
        if self.k_new.shape[0] > nd:  # the prefill chunks' tokens
            pa.pa_write_kv_paged(self.k_new[nd:], self.v_new[nd:], self.k_cache, self.v_cache, self.block_tables,
                                 self.seq_idx[nd:], self.pos[nd:], slot_mapping=self.slots[nd:],
                                 error_count=self.error_count, stream=stream)

    def decode_stage(self, stream=None):
        """Decode as the step runs it: fused with the decode tokens' KV write when possible."""
        if not self.fused_decode_write:
            return self.decode(stream)
        w, nd = self.w, self.w.num_decode
        if w.kv_fp8:
            return pa.pa_decode_write_fp8(self.q_decode, self.k_cache, self.v_cache, self.block_tables[:nd],
                                          self.context_lens[:nd], self.max_context_len, w.scale, w.k_scale, w.v_scale,
                                          self.k_new[:nd], self.v_new[:nd], self.workspace, out=self.out_decode,
                                          new_slots=self.slots[:nd], error_count=self.error_count, stream=stream)
        return pa.pa_decode_write(self.q_decode, self.k_cache, self.v_cache, self.block_tables[:nd],
                                  self.context_lens[:nd], self.max_context_len, w.scale, self.k_new[:nd],
                                  self.v_new[:nd], self.workspace, out=self.out_decode, new_slots=self.slots[:nd],
                                  error_count=self.error_count, stream=stream)

    def run(self, stream=None):
        """The whole step: write this step's K/V, then attend (the decode tokens' K/V written by the decode
        kernel itself when fused_decode_write)."""
        self.write_stage(stream)
        self.decode_stage(stream)
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

    # serving from host memory ------------------------------------------
    def pinned_inputs(self) -> torch.Tensor:
        """A pinned host copy of the packed input buffer (this step's inputs); a
        serving loop writes each step's inputs into it in the same layout."""
        return self.inbuf.cpu().pin_memory()

    def pinned_outputs(self) -> torch.Tensor:
        """A pinned host buffer the size of the packed output buffer."""
        return torch.empty(self.outbuf.shape, dtype=torch.uint8).pin_memory()

    def input_views(self, host_in: torch.Tensor) -> dict:
        """Name -> view of a packed input buffer (for filling the next step's inputs)."""
        _, views = _packed_views(host_in, [getattr(self, n) for n in STEP_INPUTS])
        return dict(zip(STEP_INPUTS, views))

    def output_views(self, host_out: torch.Tensor):
        """(decode output, prefill output) as views of a packed output buffer."""
        _, views = _packed_views(host_out, [self.out_decode, self.out_prefill])
        return views

    # outputs up to this size are stored by the step's kernels straight into pinned host memory; larger ones
    # (a prefill batch's) are written to device memory and copied out, since kernels storing tens of megabytes
    # across the host link were measured to slow down more than the copy costs
    DIRECT_OUTPUT_BYTES = 4 << 20

    def step_from_host(self, host_in: torch.Tensor, host_out: torch.Tensor, stream=None):
        """One step from pinned host memory, eagerly: the packed inputs copied in
        by a kernel reading the pinned buffer (pa_stage_copy), then the step,
        whose kernels store each small output straight into the pinned output
        buffer through its device mapping; a large output is copied out after
        the step."""
        pa.pa_stage_copy(self.inbuf, host_in, stream=stream)
        dev_out = (self.out_decode, self.out_prefill)
        host_views = self.output_views(host_out)
        direct = [t.numel() * t.element_size() <= self.DIRECT_OUTPUT_BYTES for t in dev_out]
        self.out_decode, self.out_prefill = (h if d else t for h, t, d in zip(host_views, dev_out, direct))
        try:
            self.run(stream)
        finally:
            self.out_decode, self.out_prefill = dev_out
        for h, t, d in zip(host_views, dev_out, direct):
            if not d and t.numel():
                pa.pa_stage_copy(h, t, stream=stream)
        return host_out

    def capture_from_host(self, host_in: torch.Tensor, host_out: torch.Tensor) -> "torch.cuda.CUDAGraph":
        """Record copy-in and the step (writing into host_out) as one CUDA graph
        bound to these two pinned buffers: a serving loop writes the next step's
        inputs into host_in, replays, and reads host_out once the stream is
        synchronised.  Call after one eager step."""
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.step_from_host(host_in, host_out)
        torch.cuda.current_stream(self.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step_from_host(host_in, host_out)
        self.host_graph = (g, host_in.data_ptr(), host_out.data_ptr())
        return g

    def run_from_host(self, host_in: torch.Tensor, host_out: torch.Tensor, graph: bool = True):
        """One step from pinned host memory: copy the packed inputs in and run the
        step with its outputs stored into host_out — the captured graph of
        capture_from_host when `graph` and it was captured for these buffers,
        else eagerly.  Asynchronous on the current stream."""
        hg = getattr(self, "host_graph", None)
        if graph and hg is not None and hg[1] == host_in.data_ptr() and hg[2] == host_out.data_ptr():
            hg[0].replay()
        else:
            self.step_from_host(host_in, host_out)
        return host_out

    def errors(self) -> int:
        return int(self.error_count.item()) if self.error_count is not None else 0
