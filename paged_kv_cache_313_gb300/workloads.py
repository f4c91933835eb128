"""Seeded synthetic inputs for the paged-attention hot path.

This module only *draws* inputs: sequence lengths, block placement (through the
:class:`~paged_kv_cache_313_gb300.allocator.BlockAllocator`), and N(0,1) values
for the pools, the new tokens' K/V and the queries.  It computes no slot, no
address and no attention; both the CUDA library and the CPU oracle consume what
it returns.

The five named workloads follow the serving scenarios the pages describe
(variable context lengths, grouped KV heads, shared prefixes, continuous
batching).  Every workload is one *step*: the new tokens of this step are
listed in ``seq_idx``/``pos`` with their K/V in ``k_new``/``v_new`` and must be
scattered into the pools before attention runs; ``context_lens`` already
counts them.

Pool contents: every slot of both pools starts as N(0,1) noise, so slots that no
sequence owns hold finite garbage that a correct kernel never reads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from .allocator import BlockAllocator, CowCopy
from .cascade import cascade_groups

WORKLOADS = ("tiny_fp32", "decode_bf16", "longctx_bf16", "shared_prefix_bf16", "mixed_bf16")


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    k_cache: torch.Tensor  # [P, B, Hkv, D], host, before this step's writes
    v_cache: torch.Tensor
    block_tables: torch.Tensor  # int32 [S, max_blocks_per_seq], -1 padded
    context_lens: torch.Tensor  # int32 [S]
    seq_idx: torch.Tensor  # int32 [T]  new tokens of this step
    pos: torch.Tensor  # int32 [T]
    k_new: torch.Tensor  # [T, Hkv, D]
    v_new: torch.Tensor
    num_decode: int  # rows 0..num_decode-1 of the table are decode sequences
    q_decode: torch.Tensor  # [num_decode, Hq, D]
    cu_q_lens: torch.Tensor  # int32 [C+1] chunked-prefill queries (C may be 0)
    q_start_pos: torch.Tensor  # int32 [C]
    seq_of_chunk: torch.Tensor  # int32 [C]
    q_prefill: torch.Tensor  # [total_q, Hq, D]
    cow_copies: list = field(default_factory=list)
    meta: dict = field(default_factory=dict)
    allocator: BlockAllocator | None = None  # the allocator state that produced the tables
    seq_ids: list = field(default_factory=list)  # allocator ids of the table's rows
    # decode sequences grouped by shared leading blocks (cascade.cascade_groups)
    group_offsets: torch.Tensor | None = None  # int32 [G+1]
    prefix_lens: torch.Tensor | None = None  # int32 [num_decode]
    max_group_size: int = 0
    # e4m3 pools (uint8 codes read back as code * scale); q, new K/V and outputs stay bf16
    kv_fp8: bool = False
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_seqs(self) -> int:
        return int(self.block_tables.shape[0])

    @property
    def num_chunks(self) -> int:
        return int(self.q_start_pos.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_decode_context(self) -> int:
        return int(self.context_lens[: self.num_decode].max()) if self.num_decode else 0

    @property
    def max_q_len(self) -> int:
        return int((self.cu_q_lens[1:] - self.cu_q_lens[:-1]).max()) if self.num_chunks else 0

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()

    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token across all KV heads (one layer)."""
        return 2 * self.num_kv_heads * self.head_dim * (1 if self.kv_fp8 else self.elem_bytes)


def _normal(rng: np.random.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    x = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32))
    return x.to(dtype) if dtype != torch.float32 else x


def _finish(name, dtype, Hq, Hkv, D, B, alloc: BlockAllocator, rng, decode_seqs, decode_ctx,
            chunk_seqs=(), chunk_off=(), chunk_len=(), cow=(), scale=None, meta=None) -> Workload:
    P = alloc.num_blocks
    seqs = list(decode_seqs) + list(chunk_seqs)
    width = max(alloc.blocks_for(alloc.seq_len(s)) for s in seqs)
    bt = torch.from_numpy(alloc.block_table(seqs, width))
    ctx = torch.tensor([alloc.seq_len(s) for s in seqs], dtype=torch.int32)
    assert list(ctx[: len(decode_seqs)]) == list(decode_ctx)
    k_cache = _normal(rng, (P, B, Hkv, D), dtype)
    v_cache = _normal(rng, (P, B, Hkv, D), dtype)
    for c in cow:  # copy-on-write copies are applied to the pool as the allocator requested them
        k_cache[c.dst, : c.num_valid] = k_cache[c.src, : c.num_valid]
        v_cache[c.dst, : c.num_valid] = v_cache[c.src, : c.num_valid]
    nd = len(decode_seqs)
    seq_idx = list(range(nd))
    pos = [int(L) - 1 for L in decode_ctx]
    cu = [0]
    for i, (off, n) in enumerate(zip(chunk_off, chunk_len)):
        seq_idx += [nd + i] * n
        pos += list(range(off, off + n))
        cu.append(cu[-1] + n)
    T = len(seq_idx)
    k_new = _normal(rng, (T, Hkv, D), dtype)
    v_new = _normal(rng, (T, Hkv, D), dtype)
    q_decode = _normal(rng, (nd, Hq, D), dtype)
    q_prefill = _normal(rng, (cu[-1], Hq, D), dtype)
    goff, pre, gmax = cascade_groups(bt[:nd].numpy(), ctx[:nd].numpy(), B, max_members=max(1, 32 // (Hq // Hkv)))
    return Workload(
        name=name, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B, num_blocks=P,
        scale=scale if scale is not None else 1.0 / math.sqrt(D),
        k_cache=k_cache, v_cache=v_cache, block_tables=bt, context_lens=ctx,
        seq_idx=torch.tensor(seq_idx, dtype=torch.int32), pos=torch.tensor(pos, dtype=torch.int32),
        k_new=k_new, v_new=v_new, num_decode=nd, q_decode=q_decode,
        cu_q_lens=torch.tensor(cu, dtype=torch.int32),
        q_start_pos=torch.tensor(list(chunk_off), dtype=torch.int32),
        seq_of_chunk=torch.tensor([nd + i for i in range(len(chunk_off))], dtype=torch.int32),
        q_prefill=q_prefill, cow_copies=list(cow), meta=dict(meta or {}), allocator=alloc, seq_ids=seqs,
        group_offsets=torch.from_numpy(goff), prefix_lens=torch.from_numpy(pre), max_group_size=gmax)


def _pool_size(needed_blocks: int, spare: float = 0.10) -> int:
    return int(math.ceil((1.0 + spare) * needed_blocks))


def _decode_batch(name, lens, Hq, Hkv, D, B, dtype, seed, num_blocks=None, scale=None, meta=None):
    lens = [int(L) for L in lens]
    rng = np.random.default_rng(seed)
    needed = sum(-(-L // B) for L in lens)
    alloc = BlockAllocator(num_blocks or _pool_size(needed), B, seed=seed + 1)
    seqs = []
    for L in lens:
        s = alloc.allocate(L - 1)  # history already in the pool
        alloc.append(s, 1)  # this step's token (may open a new block)
        seqs.append(s)
    return _finish(name, dtype, Hq, Hkv, D, B, alloc, rng, seqs, lens, scale=scale, meta=meta)


def tiny_fp32(seed: int = 0) -> Workload:
    """4 sequences, lengths {1, 16, 17, 40}, 4/4 heads, D=64, B=16, pool of 64 blocks, fp32."""
    return _decode_batch("tiny_fp32", [1, 16, 17, 40], 4, 4, 64, 16, torch.float32, seed, num_blocks=64,
                         scale=1.0 / 8.0)


def decode_bf16(seed: int = 0, num_seqs: int = 64, min_len: int = 128, max_len: int = 4096) -> Workload:
    """64 sequences, lengths U[128, 4096], 32/8 heads, D=128, B=16, pool = needed + 10%, bf16."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(min_len, max_len, size=num_seqs, endpoint=True)
    return _decode_batch("decode_bf16", lens, 32, 8, 128, 16, torch.bfloat16, seed)


def longctx_bf16(seed: int = 0, num_seqs: int = 16, min_len: int = 1024, max_len: int = 32768) -> Workload:
    """16 sequences, lengths log-uniform in [1024, 32768], 64/8 heads, D=128, B=16, bf16."""
    rng = np.random.default_rng(seed + 2000)
    lens = np.rint(np.exp(rng.uniform(math.log(min_len), math.log(max_len), size=num_seqs))).astype(np.int64)
    lens = np.clip(lens, min_len, max_len)
    return _decode_batch("longctx_bf16", lens, 64, 8, 128, 16, torch.bfloat16, seed)


def shared_prefix_bf16(seed: int = 0, num_prompts: int = 32, branches: int = 8, prefix_len: int = 2048,
                       max_tail: int = 512, B: int = 16, name: str = "shared_prefix_bf16", num_q_heads: int = 32,
                       num_kv_heads: int = 8) -> Workload:
    """Parallel sampling: each prompt's prefix blocks are shared (ref-counted) by its
    branches; each branch then adds a private tail of U{0..max_tail} tokens and one
    new token.  A prefix that ends inside a block makes each branch's first write
    copy the shared partial block (copy-on-write)."""
    rng = np.random.default_rng(seed + 3000)
    tails = rng.integers(0, max_tail, size=(num_prompts, branches), endpoint=True)
    prefix_blocks = -(-prefix_len // B)
    private = sum(-(-(prefix_len + int(t) + 1) // B) - prefix_len // B for t in tails.ravel())
    alloc = BlockAllocator(_pool_size(num_prompts * prefix_blocks + private), B, seed=seed + 1)
    seqs, lens, cow = [], [], []
    for p in range(num_prompts):
        root = alloc.allocate(prefix_len)
        kids = [alloc.fork(root) for _ in range(branches)]
        alloc.free(root)  # the prefix is now referenced by the branches only
        for b, s in enumerate(kids):
            t = int(tails[p, b])
            if t:
                cow += alloc.append(s, t)  # private tail history
            cow += alloc.append(s, 1)  # this step's token
            seqs.append(s)
            lens.append(prefix_len + t + 1)
    vrng = np.random.default_rng(seed)
    meta = {"prefix_len": prefix_len, "num_prompts": num_prompts, "branches": branches,
            "unique_tokens": num_prompts * prefix_len + int(tails.sum()) + num_prompts * branches}
    return _finish(name, torch.bfloat16, num_q_heads, num_kv_heads, 128, B, alloc, vrng, seqs, lens, cow=cow,
                   meta=meta)


def as_fp8(w: Workload, seed: int, k_scale: float = 1.0 / 64, v_scale: float = 1.0 / 64, lo: int = 0x30,
           hi: int = 0x60) -> Workload:
    """The same batch over e4m3 pools: every pool byte becomes a random code whose low seven bits are drawn
    from [lo, hi) (0x30..0x5f: exponent fields 6..11, magnitudes 0.25..60 before the scale; hi <= 0x7f keeps
    NaN codes out) with a random sign.  Queries and the new tokens' K/V stay bf16."""
    rng = np.random.default_rng(seed + 5000)
    shape = tuple(w.k_cache.shape)
    codes = lambda: torch.from_numpy(rng.integers(lo, hi, size=shape, dtype=np.uint8) |  # noqa: E731
                                     (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7))
    w.k_cache, w.v_cache = codes(), codes()
    w.kv_fp8, w.k_scale, w.v_scale = True, float(k_scale), float(v_scale)
    return w


def decode_fp8(seed: int = 0, num_seqs: int = 64, min_len: int = 128, max_len: int = 4096) -> Workload:
    """The bf16 decode workload's batch (64 sequences, lengths U[128, 4096], 32/8 heads, D=128, B=16) over e4m3
    pools (history codes as in ``as_fp8``, k_scale = v_scale = 1/64)."""
    w = as_fp8(decode_bf16(seed, num_seqs, min_len, max_len), seed)
    w.name = "decode_fp8"
    return w


def shared_prefix_cow_bf16(seed: int = 0) -> Workload:
    """Correctness variant of the shared-prefix workload whose 2050-token prefix
    ends two tokens into a block, so the branches' first writes copy it."""
    return shared_prefix_bf16(seed, num_prompts=4, branches=8, prefix_len=2050, max_tail=40,
                              name="shared_prefix_cow_bf16")


def mixed_bf16(seed: int = 0, num_decode: int = 256, num_chunks: int = 4, chunk_len: int = 512,
               max_off: int = 4096, B: int = 32) -> Workload:
    """Continuous-batching step: decode sequences with lognormal lengths (median 1024,
    sigma 1, clipped to [16, 16384]) plus chunked-prefill requests of ``chunk_len``
    queries at prior offsets U{0..max_off}; B=32."""
    rng = np.random.default_rng(seed + 4000)
    lens = np.clip(np.rint(1024.0 * np.exp(rng.standard_normal(num_decode))), 16, 16384).astype(np.int64)
    offs = rng.integers(0, max_off, size=num_chunks, endpoint=True)
    needed = sum(-(-int(L) // B) for L in lens) + sum(-(-(int(o) + chunk_len) // B) for o in offs)
    alloc = BlockAllocator(_pool_size(needed), B, seed=seed + 1)
    dseqs = []
    for L in lens:
        s = alloc.allocate(int(L) - 1)
        alloc.append(s, 1)
        dseqs.append(s)
    cseqs = []
    for o in offs:
        s = alloc.allocate(int(o))  # history before the chunk
        alloc.append(s, chunk_len)  # the chunk's own tokens, written this step
        cseqs.append(s)
    vrng = np.random.default_rng(seed)
    return _finish("mixed_bf16", torch.bfloat16, 32, 8, 128, B, alloc, vrng, dseqs, [int(L) for L in lens],
                   chunk_seqs=cseqs, chunk_off=[int(o) for o in offs], chunk_len=[chunk_len] * num_chunks)


def prefill_batch(seed: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int, chunk_lens,
                  offsets, dtype: torch.dtype = torch.bfloat16, decode_lens=()) -> Workload:
    """A batch of chunked-prefill requests (chunk c: ``chunk_lens[c]`` queries at
    prior offset ``offsets[c]``), optionally with decode sequences, for any head
    layout and block size."""
    B = block_size
    needed = sum(-(-int(L) // B) for L in decode_lens) + sum(-(-(int(o) + int(n)) // B)
                                                          for o, n in zip(offsets, chunk_lens))
    alloc = BlockAllocator(_pool_size(max(needed, 1)) + 4, B, seed=seed + 1)
    dseqs = []
    for L in decode_lens:
        s = alloc.allocate(int(L) - 1)
        alloc.append(s, 1)
        dseqs.append(s)
    cseqs = []
    for o, n in zip(offsets, chunk_lens):
        s = alloc.allocate(int(o))
        alloc.append(s, int(n))
        cseqs.append(s)
    vrng = np.random.default_rng(seed)
    return _finish(f"prefill_g{num_q_heads // num_kv_heads}_b{B}", dtype, num_q_heads, num_kv_heads, head_dim, B,
                   alloc, vrng, dseqs, [int(L) for L in decode_lens], chunk_seqs=cseqs,
                   chunk_off=[int(o) for o in offsets], chunk_len=[int(n) for n in chunk_lens])


def small(name: str, seed: int = 0) -> Workload:
    """Reduced-size versions of the bf16 workloads (same shapes per token, fewer and
    shorter sequences) for quick parity runs that still span several tiles and
    ragged tails."""
    if name == "decode_bf16":
        return decode_bf16(seed, num_seqs=12, min_len=1, max_len=700)
    if name == "longctx_bf16":
        return longctx_bf16(seed, num_seqs=4, min_len=900, max_len=5000)
    if name == "shared_prefix_bf16":
        return shared_prefix_bf16(seed, num_prompts=3, branches=4, prefix_len=256, max_tail=40)
    if name == "mixed_bf16":
        return mixed_bf16(seed, num_decode=12, num_chunks=3, chunk_len=200, max_off=500)
    if name == "tiny_fp32":
        return tiny_fp32(seed)
    if name == "decode_fp8":
        return decode_fp8(seed, num_seqs=12, min_len=1, max_len=700)
    raise KeyError(name)


def make(name: str, seed: int = 0) -> Workload:
    return {"tiny_fp32": tiny_fp32, "decode_bf16": decode_bf16, "longctx_bf16": longctx_bf16,
            "shared_prefix_bf16": shared_prefix_bf16, "shared_prefix_cow_bf16": shared_prefix_cow_bf16,
            "mixed_bf16": mixed_bf16, "decode_fp8": decode_fp8}[name](seed)


def storage_numpy(t: torch.Tensor) -> np.ndarray:
    """Host numpy view in storage form: float32 stays float32, bf16 becomes its uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    return t.numpy()
