"""GB300-native paged-attention hot path: slot mapping, paged KV write, split-KV
paged decode and causal chunked prefill, as hand-written sm_103a CUDA behind a
C ABI (``libpa.so``), with a host-side block allocator and seeded workloads.

Importing the package needs no GPU.  The CUDA entry points live in
:mod:`paged_kv_cache_313_gb300.pa`; they raise if the library was not built or
cannot be loaded — there is no CPU fallback.
"""
from .allocator import BlockAllocator, CowCopy, NoBlocks  # noqa: F401

__all__ = ["BlockAllocator", "CowCopy", "NoBlocks"]
