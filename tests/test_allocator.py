"""Host block allocator: block counts, tail waste, placement, reference counts,
copy-on-write and explicit failure on exhaustion."""
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_313_gb300.allocator import BlockAllocator, NoBlocks


def test_worked_example_counts(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example_b16.json")))
    a = BlockAllocator(64, g["block_size"], seed=0)
    s = a.allocate(g["seq_len"])
    assert len(a.blocks(s)) == g["num_blocks"]
    s17 = a.allocate(g["len17"]["seq_len"])
    assert len(a.blocks(s17)) == g["len17"]["num_blocks"]
    ex = g["kv_tokens_example"]
    big = BlockAllocator(400, 16, seed=1)
    p = big.allocate(ex["prompt"])
    for _ in range(ex["generated"]):
        big.append(p, 1)
    assert big.seq_len(p) == ex["total"]
    assert len(big.blocks(p)) == oracle.num_blocks(ex["total"], 16)
    big.check_invariants()


@pytest.mark.parametrize("B", [1, 2, 16, 32])
def test_block_count_matches_oracle_and_tail_waste(B):
    a = BlockAllocator(5000, B, seed=3)
    for L in range(0, 200):
        s = a.allocate(L)
        n = len(a.blocks(s))
        assert n == oracle.num_blocks(L, B)
        assert 0 <= n * B - L <= B - 1
        a.free(s)
    a.check_invariants()
    assert a.num_free == 5000


def test_decode_appends_fill_tail_before_new_block():
    a = BlockAllocator(32, 16, seed=0)
    s = a.allocate(15)
    assert len(a.blocks(s)) == 1
    a.append(s)  # 16th token fills the tail
    assert len(a.blocks(s)) == 1
    a.append(s)  # 17th opens block 2
    assert len(a.blocks(s)) == 2
    for _ in range(15):
        a.append(s)
    assert len(a.blocks(s)) == 2 and a.seq_len(s) == 32
    a.check_invariants()


def test_random_noncontiguous_placement():
    a = BlockAllocator(1000, 16, seed=7)
    s = a.allocate(16 * 50)
    blocks = np.array(a.blocks(s))
    assert len(set(blocks.tolist())) == 50
    assert np.count_nonzero(np.diff(blocks) == 1) < 10  # not laid out contiguously
    b = BlockAllocator(1000, 16, seed=7)
    assert b.blocks(b.allocate(16 * 50)) == blocks.tolist()  # seeded: reproducible


def test_refcount_lifecycle_and_fork():
    a = BlockAllocator(20, 4, seed=0)
    root = a.allocate(10)  # 3 blocks
    kids = [a.fork(root) for _ in range(3)]
    assert all(a.ref_cnt[b] == 4 for b in a.blocks(root))
    a.free(root)
    assert all(a.ref_cnt[b] == 3 for b in a.blocks(kids[0]))
    a.free(kids[0])
    a.free(kids[1])
    assert a.num_free == 17
    a.free(kids[2])
    assert a.num_free == 20 and np.all(a.ref_cnt == 0)
    a.check_invariants()


def test_copy_on_write_shared_partial_block():
    a = BlockAllocator(20, 4, seed=0)
    root = a.allocate(10)  # blocks: full, full, partial (2 valid)
    k1, k2 = a.fork(root), a.fork(root)
    a.free(root)
    shared = a.blocks(k1)
    tail = shared[-1]
    copies = a.append(k1, 1)
    assert len(copies) == 1
    c = copies[0]
    assert c.src == tail and c.num_valid == 2 and c.dst not in shared
    assert a.blocks(k1)[:-1] == shared[:-1] and a.blocks(k1)[-1] == c.dst
    assert a.blocks(k2) == shared  # the other branch is untouched
    assert a.ref_cnt[tail] == 1 and a.ref_cnt[c.dst] == 1
    # the last holder of the partial block writes in place: no copy
    assert a.append(k2, 1) == []
    assert a.blocks(k2) == shared
    # full shared blocks are never copied: a new block opens on the boundary
    r2 = a.allocate(8)
    k3, k4 = a.fork(r2), a.fork(r2)
    a.free(r2)
    assert a.append(k3, 1) == [] and len(a.blocks(k3)) == 3 and a.blocks(k3)[:2] == a.blocks(k4)
    a.check_invariants()


def test_exhaustion_is_explicit_and_mutates_nothing():
    a = BlockAllocator(4, 4, seed=0)
    s = a.allocate(12)  # 3 blocks, 1 free
    other = a.fork(s)
    snapshot = (a.blocks(s), a.blocks(other), a.ref_cnt.copy(), a.num_free)
    with pytest.raises(NoBlocks):
        a.allocate(8)
    with pytest.raises(NoBlocks):
        a.append(s, 5)  # needs 2 blocks
    assert (a.blocks(s), a.blocks(other), a.num_free) == snapshot[:2] + (snapshot[3],)
    assert np.array_equal(a.ref_cnt, snapshot[2]) and a.seq_len(s) == 12
    a.check_invariants()
    a.append(s, 4)  # exactly one block: fine
    with pytest.raises(NoBlocks):
        a.append(s, 1)
    a.check_invariants()


def test_cow_exhaustion_mutates_nothing():
    a = BlockAllocator(3, 4, seed=0)
    root = a.allocate(6)  # 2 blocks, partial tail
    k1 = a.fork(root)
    a.allocate(1)  # take the last free block
    with pytest.raises(NoBlocks):
        a.append(k1, 1)  # would need a private copy of the shared tail
    assert a.blocks(k1) == a.blocks(root) and a.seq_len(k1) == 6
    a.check_invariants()


def test_block_table_export():
    a = BlockAllocator(50, 16, seed=0)
    s1, s2 = a.allocate(40), a.allocate(1)
    bt = a.block_table([s1, s2])
    assert bt.dtype == np.int32 and bt.shape == (2, 3)
    assert bt[0].tolist() == a.blocks(s1) and bt[1, 0] == a.blocks(s2)[0] and bt[1, 1:].tolist() == [-1, -1]
    with pytest.raises(ValueError):
        a.block_table([s1], max_blocks_per_seq=2)
