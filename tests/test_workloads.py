"""Seeded workload generator: shapes, lengths and table structure of the five
workloads, and that every table row covers exactly its context."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_313_gb300 import workloads as W


def _check_tables(w):
    bt = w.block_tables.numpy()
    ctx = w.context_lens.numpy()
    for s in range(w.num_seqs):
        n = oracle.num_blocks(int(ctx[s]), w.block_size)
        assert np.all(bt[s, :n] >= 0) and np.all(bt[s, :n] < w.num_blocks)
        assert np.all(bt[s, n:] == -1)


def test_tiny_fp32_matches_spec():
    w = W.tiny_fp32(0)
    assert w.context_lens.tolist() == [1, 16, 17, 40]
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks) == (4, 4, 64, 16, 64)
    assert w.dtype == torch.float32 and math.isclose(w.scale, 1 / math.sqrt(64))
    assert w.pos.tolist() == [0, 15, 16, 39] and w.seq_idx.tolist() == [0, 1, 2, 3]
    used = w.block_tables[w.block_tables >= 0]
    assert used.numel() == 7 and len(set(used.tolist())) == 7
    # KV bytes = layers x tokens x kv_heads x head_dim x 2 x dtype_size (one layer, whole pool)
    assert w.k_cache.nbytes + w.v_cache.nbytes == 1 * 64 * 16 * 4 * 64 * 2 * 4
    _check_tables(w)


def test_decode_bf16_matches_spec():
    w = W.decode_bf16(0)
    ctx = w.context_lens.numpy()
    assert w.num_seqs == 64 and ctx.min() >= 128 and ctx.max() <= 4096
    needed = sum(oracle.num_blocks(int(L), 16) for L in ctx)
    assert w.num_blocks == math.ceil(1.1 * needed)
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.dtype) == (32, 8, 128, 16, torch.bfloat16)
    _check_tables(w)
    assert W.decode_bf16(0).context_lens.tolist() == ctx.tolist()  # seeded


def test_longctx_lengths_loguniform_range():
    w = W.longctx_bf16(0)
    ctx = w.context_lens.numpy()
    assert w.num_seqs == 16 and ctx.min() >= 1024 and ctx.max() <= 32768
    assert (w.num_q_heads, w.num_kv_heads) == (64, 8)
    _check_tables(w)


def test_shared_prefix_structure():
    w = W.shared_prefix_bf16(0)
    bt = w.block_tables.numpy()
    assert w.num_seqs == 256
    for p in range(32):
        rows = bt[p * 8:(p + 1) * 8, :128]
        assert np.all(rows == rows[0])  # 128 shared full prefix blocks per prompt
    assert len({tuple(bt[p * 8, :128]) for p in range(32)}) == 32
    assert w.cow_copies == []  # a 2048-token prefix ends on a block boundary
    _check_tables(w)


def test_shared_prefix_cow_variant_copies_partial_block():
    w = W.shared_prefix_cow_bf16(0)
    assert len(w.cow_copies) == 4 * 7  # every branch but the last holder copies the partial block
    for c in w.cow_copies:
        assert c.num_valid == 2
        assert torch.equal(w.k_cache[c.dst, :2], w.k_cache[c.src, :2])
        assert torch.equal(w.v_cache[c.dst, :2], w.v_cache[c.src, :2])
    _check_tables(w)


def test_mixed_structure():
    w = W.small("mixed_bf16")
    assert w.num_chunks == 3 and w.block_size == 32
    ctx = w.context_lens.numpy()
    for c in range(w.num_chunks):
        s = int(w.seq_of_chunk[c])
        n = int(w.cu_q_lens[c + 1] - w.cu_q_lens[c])
        assert ctx[s] == int(w.q_start_pos[c]) + n
    assert w.seq_idx.numel() == w.num_decode + int(w.cu_q_lens[-1])
    _check_tables(w)


@pytest.mark.parametrize("name", ["decode_bf16", "longctx_bf16", "shared_prefix_bf16", "mixed_bf16"])
def test_small_variants(name):
    _check_tables(W.small(name))
