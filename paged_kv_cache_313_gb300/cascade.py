"""Host-side grouping for cascade decode (``pa_decode_cascade``).

Sequences forked from a common parent keep mapping the parent's physical
blocks ("什么是 PagedAttention？", 共享但不污染状态: shared blocks are
reference-counted and copied only when a sharer writes).  Decode can read
such a shared prefix once per group instead of once per sequence.  This module
finds the groups from the block tables alone: a group is a maximal run of
consecutive sequences whose tables start with the same physical blocks, and
its prefix is the tokens those common leading blocks hold (capped by every
member's context).  Blocks that were copied on write are private, so a copied
partial block falls to each member's own tail.
"""
from __future__ import annotations

import numpy as np


def cascade_groups(block_tables, context_lens, block_size: int, num_seqs: int | None = None,
                   max_members: int | None = None):
    """Return (group_offsets int32 [G+1], prefix_lens int32 [N], max_group_size).

    block_tables: int [N, W] (rows beyond a sequence's blocks are ignored);
    context_lens: int [N].  Every sequence lands in exactly one group; a group
    of one has prefix 0.  A run longer than max_members is cut into groups of
    at most max_members (the decode kernel reads a group's queries as one tile
    of at most 32 rows: max_members = 32 // (query heads per kv head)).
    """
    bt = np.asarray(block_tables)
    ctx = np.asarray(context_lens).astype(np.int64)
    n = int(ctx.shape[0] if num_seqs is None else num_seqs)
    nblk = -(-ctx[:n] // block_size)
    offsets, prefix = [0], np.zeros(n, dtype=np.int32)
    s = 0
    while s < n:
        e = s + 1
        common = int(nblk[s])  # leading blocks the run shares with its first member
        while (common > 0 and e < n and nblk[e] > 0 and bt[e, 0] == bt[s, 0]
               and (max_members is None or e - s < max_members)):
            k = min(common, int(nblk[e]))
            same = bt[s, :k] == bt[e, :k]
            common = k if same.all() else int(np.argmin(same))  # >= 1: the first blocks match
            e += 1
        if e - s > 1 and common > 0:
            prefix[s:e] = min(common * block_size, int(ctx[s:e].min()))
        offsets.append(e)
        s = e
    sizes = np.diff(offsets)
    return np.asarray(offsets, dtype=np.int32), prefix, int(sizes.max()) if len(sizes) else 0
