"""Host-side grouping for cascade decode: which consecutive decode sequences
share leading physical blocks, and how many tokens those blocks cover."""
import numpy as np

from paged_kv_cache_313_gb300 import workloads as W
from paged_kv_cache_313_gb300.cascade import cascade_groups


def test_hand_made_tables():
    # seqs 0-2 share block 5; 0 and 1 also share 6; seq 3 shares nothing
    bt = np.array([[5, 6, 7], [5, 6, 9], [5, 8, 1], [2, 3, 4]], np.int32)
    ctx = np.array([40, 45, 33, 20], np.int32)
    off, pre, mx = cascade_groups(bt, ctx, 16)
    assert off.tolist() == [0, 3, 4] and mx == 3
    assert pre.tolist() == [16, 16, 16, 0]  # one common block for all three members


def test_prefix_capped_by_the_shortest_member():
    bt = np.array([[4, 5, -1], [4, 5, 6]], np.int32)
    ctx = np.array([20, 40], np.int32)  # member 0 has only 20 tokens: 4 of block 5
    off, pre, _ = cascade_groups(bt, ctx, 16)
    assert off.tolist() == [0, 2] and pre.tolist() == [20, 20]


def test_shared_prefix_workloads():
    w = W.small("shared_prefix_bf16", 0)  # 3 prompts x 4 branches, 256-token prefix
    assert w.group_offsets.tolist() == [0, 4, 8, 12] and w.max_group_size == 4
    assert set(w.prefix_lens.tolist()) == {256}
    # a 2050-token prefix ends 2 tokens into a block that each branch copied on write: only the
    # 128 full blocks stay shared, the copied partial block belongs to every member's own tail
    w = W.make("shared_prefix_cow_bf16", 0)
    assert set(w.prefix_lens.tolist()) == {2048}
    nd = w.num_decode
    for g in range(len(w.group_offsets) - 1):
        a, b = int(w.group_offsets[g]), int(w.group_offsets[g + 1])
        P = int(w.prefix_lens[a])
        tables = w.block_tables[a:b, : P // w.block_size]
        assert (tables == tables[0]).all()
        assert int(w.context_lens[a:b].min()) > P
    assert int(w.group_offsets[-1]) == nd


def test_unshared_batches_are_singletons():
    w = W.small("decode_bf16", 0)
    assert w.group_offsets.tolist() == list(range(w.num_decode + 1))
    assert int(w.prefix_lens.max()) == 0 and w.max_group_size == 1


def test_runs_longer_than_the_tile_are_cut():
    bt = np.array([[7, 8]] * 5 + [[1, 2]], np.int32)
    ctx = np.array([30] * 5 + [30], np.int32)
    off, pre, mx = cascade_groups(bt, ctx, 16, max_members=2)
    assert off.tolist() == [0, 2, 4, 5, 6] and mx == 2
    assert pre.tolist() == [30, 30, 30, 30, 0, 0]  # a group of one keeps no prefix
