"""Memory-utilisation measurements against the pages' worked numbers."""
import json
import os

import pytest

from paged_kv_cache_313_gb300.allocator import BlockAllocator
from paged_kv_cache_313_gb300.memstats import kv_bytes_per_token, utilisation


def test_worked_example_fragmentation_and_tail(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example_b16.json")))
    a = BlockAllocator(64, g["block_size"], seed=0)
    s = a.allocate(g["seq_len"])
    u = utilisation(a, [s], bytes_per_token=1)
    assert u["unique_blocks"] == g["num_blocks"] and u["used_slots"] == g["seq_len"]
    assert u["fragmentation"] == pytest.approx(1 - 40 / 48)
    assert u["max_tail_waste_slots"] <= g["max_tail_waste"]


def test_reservation_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example_b16.json")))["reservation_example"]
    a = BlockAllocator(64, 16, seed=0)
    s = a.allocate(g["used"])
    u = utilisation(a, [s], bytes_per_token=1, max_len=g["reserved"])
    assert u["contiguous_reserved_bytes"] - u["used_slots"] == g["wasted"]
    assert u["fragmentation"] == 0.0  # 512 fills 32 blocks exactly


def test_shared_blocks_counted_once():
    a = BlockAllocator(100, 16, seed=1)
    root = a.allocate(40)
    kids = [a.fork(root) for _ in range(4)]
    a.free(root)
    for k in kids:
        a.append(k, 1)  # copy-on-write of the shared partial block
    u = utilisation(a, kids, bytes_per_token=kv_bytes_per_token(8, 128, 2))
    assert u["unique_blocks"] == 2 + 4  # 2 shared full blocks + 4 private tails (3 copies + 1 in place)
    assert u["logical_tokens"] == 4 * 41 and u["used_slots"] == 32 + 4 * 9
    assert u["per_request_bytes_mean"] == 3 * 16 * 4096
    assert kv_bytes_per_token(8, 128, 2) == 4096
