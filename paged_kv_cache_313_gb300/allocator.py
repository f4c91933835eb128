"""Host-side block allocator: the physical block pool, block tables, reference
counts and copy-on-write.

Follows the pages' description of the block manager:

* "什么是 PagedAttention？", 工作原理 › 映射逻辑块与物理块: prefill takes blocks
  for the input length; decode appends to the partially filled tail block and
  takes a new block only once the tail is full; an allocation that cannot be
  satisfied fails explicitly and never overwrites another sequence's state.
* same page, 共享但不污染状态: sequences share immutable prefix blocks, a
  reference count decides when a block is reclaimed, and a write into a shared
  partial block first copies the valid entries into a private block and updates
  only that sequence's block table (copy-on-write).
* "PagedAttention学习笔记", §2.1 (引用计数 and the state diagram): allocate /
  touch increments ``ref_cnt``; free decrements it and a block whose count
  reaches zero returns to the free pool.
* "KV cache 显存管理：为什么 PagedAttention 是 vLLM 的核心", "Block manager 是
  PagedAttention 的前置条件": keep the free blocks, allocate for new requests,
  append on decode, keep each sequence's block table, free on finish, and
  answer whether the pool can take more work.

Placement is random and non-contiguous: the free list starts as a seeded
random permutation of the pool, so logically adjacent blocks land anywhere.
The allocator only decides *which* physical block backs each logical block; it
touches no K/V data.  Copies that copy-on-write requires are returned to the
caller as ``(src_block, dst_block, num_valid)`` records.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


class NoBlocks(RuntimeError):
    """The pool cannot satisfy an allocation.  The allocator state is unchanged."""


@dataclass
class CowCopy:
    """Copy the first ``num_valid`` token slots of ``src`` into ``dst``."""

    src: int
    dst: int
    num_valid: int


@dataclass
class _Seq:
    blocks: list = field(default_factory=list)
    length: int = 0


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int, seed: int = 0):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        rng = np.random.default_rng(seed)
        # Stack of free blocks; pop() takes the next one.  Reversed so that the
        # first allocations follow the permutation's order.
        self._free = [int(b) for b in rng.permutation(self.num_blocks)[::-1]]
        self.ref_cnt = np.zeros(self.num_blocks, dtype=np.int64)
        self._seqs: dict[int, _Seq] = {}
        self._next_id = 0

    # ------------------------------------------------------------ queries
    @property
    def num_free(self) -> int:
        return len(self._free)

    def blocks_for(self, num_tokens: int) -> int:
        """Blocks needed to hold ``num_tokens`` tokens: ceil(num_tokens / B)."""
        return -(-int(num_tokens) // self.block_size) if num_tokens > 0 else 0

    def seq_len(self, seq: int) -> int:
        return self._seqs[seq].length

    def blocks(self, seq: int) -> list:
        return list(self._seqs[seq].blocks)

    def sequences(self) -> list:
        return list(self._seqs)

    def can_allocate(self, num_blocks: int) -> bool:
        return num_blocks <= len(self._free)

    # ---------------------------------------------------------- mutations
    def _take(self, n: int) -> list:
        if n > len(self._free):
            raise NoBlocks(f"need {n} blocks, {len(self._free)} free")
        out = [self._free.pop() for _ in range(n)]
        for b in out:
            assert self.ref_cnt[b] == 0
            self.ref_cnt[b] = 1
        return out

    def _release(self, block: int) -> None:
        assert self.ref_cnt[block] > 0
        self.ref_cnt[block] -= 1
        if self.ref_cnt[block] == 0:
            self._free.append(int(block))

    def allocate(self, num_tokens: int) -> int:
        """Prefill: a new sequence holding ``num_tokens`` tokens.  Returns its id."""
        blocks = self._take(self.blocks_for(num_tokens))
        sid = self._next_id
        self._next_id += 1
        self._seqs[sid] = _Seq(blocks=blocks, length=int(num_tokens))
        return sid

    def append(self, seq: int, num_tokens: int = 1) -> list:
        """Grow ``seq`` by ``num_tokens`` tokens (decode appends one at a time).

        Fills the tail block first and takes a new block only on a block
        boundary.  Before the first write into a tail block that other
        sequences still reference, the tail is copied into a private block
        (copy-on-write).  Returns the copies the caller must perform.  On
        exhaustion raises NoBlocks and leaves every sequence unchanged.
        """
        s = self._seqs[seq]
        B = self.block_size
        new_len = s.length + int(num_tokens)
        grow = self.blocks_for(new_len) - len(s.blocks)
        tail_partial = s.length % B != 0
        cow = num_tokens > 0 and tail_partial and self.ref_cnt[s.blocks[-1]] > 1
        if grow + (1 if cow else 0) > len(self._free):
            raise NoBlocks(f"need {grow + int(cow)} blocks, {len(self._free)} free")
        copies = []
        if cow:
            src = s.blocks[-1]
            (dst,) = self._take(1)
            copies.append(CowCopy(src=src, dst=dst, num_valid=s.length % B))
            self._release(src)
            s.blocks[-1] = dst
        s.blocks.extend(self._take(grow))
        s.length = new_len
        return copies

    def fork(self, parent: int) -> int:
        """A new sequence sharing every block of ``parent`` (ref_cnt += 1 each)."""
        p = self._seqs[parent]
        for b in p.blocks:
            self.ref_cnt[b] += 1
        sid = self._next_id
        self._next_id += 1
        self._seqs[sid] = _Seq(blocks=list(p.blocks), length=p.length)
        return sid

    def free(self, seq: int) -> None:
        """Finish ``seq``: drop one reference to each of its blocks."""
        s = self._seqs.pop(seq)
        for b in s.blocks:
            self._release(b)

    # ------------------------------------------------------------ export
    def block_table(self, seqs, max_blocks_per_seq: int | None = None) -> np.ndarray:
        """int32 block table [len(seqs), max_blocks_per_seq], padded with -1."""
        rows = [self._seqs[s].blocks for s in seqs]
        width = max_blocks_per_seq if max_blocks_per_seq is not None else max((len(r) for r in rows), default=0)
        width = max(int(width), 1)
        bt = np.full((len(rows), width), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            if len(r) > width:
                raise ValueError(f"sequence needs {len(r)} blocks, table has {width} columns")
            bt[i, : len(r)] = r
        return bt

    def check_invariants(self) -> None:
        """Every block is either free with ref 0, or referenced exactly ref_cnt times."""
        counts = np.zeros(self.num_blocks, dtype=np.int64)
        for s in self._seqs.values():
            assert len(s.blocks) == self.blocks_for(s.length)
            for b in s.blocks:
                counts[b] += 1
        assert np.array_equal(counts, self.ref_cnt), "ref_cnt disagrees with the block tables"
        free = np.zeros(self.num_blocks, dtype=bool)
        free[self._free] = True
        assert len(set(self._free)) == len(self._free), "a block is on the free list twice"
        assert np.all(free == (self.ref_cnt == 0)), "free list disagrees with ref_cnt"
