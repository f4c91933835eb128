"""Expected results of one hot-path step, computed by the CPU oracle only.

Takes a seeded Workload (host tensors), runs the oracle's slot mapping, KV
write, decode and prefill on numpy copies, and returns everything the GPU path
must reproduce.  Nothing here touches the CUDA library.
"""
from dataclasses import dataclass

import numpy as np

import oracle
from paged_kv_cache_313_gb300.workloads import Workload, storage_numpy


@dataclass
class Expected:
    slots: np.ndarray
    slot_errors: int
    k_cache: np.ndarray  # storage form, after this step's writes
    v_cache: np.ndarray
    out_decode: np.ndarray | None  # fp64
    out_prefill: np.ndarray | None


def expected_step(w: Workload, attention: bool = True, threads: int = 0) -> Expected:
    bt = w.block_tables.numpy()
    slots, err = oracle.slot_mapping(bt, w.seq_idx.numpy(), w.pos.numpy(), w.block_size, w.num_blocks)
    kc = storage_numpy(w.k_cache).copy()
    vc = storage_numpy(w.v_cache).copy()
    if w.kv_fp8:  # e4m3 pools: the quantising write, then attention on the read-back values (float64)
        werr = oracle.write_kv_fp8(storage_numpy(w.k_new), storage_numpy(w.v_new), kc, vc, slots, w.k_scale,
                                   w.v_scale)
    else:
        werr = oracle.write_kv(storage_numpy(w.k_new), storage_numpy(w.v_new), kc, vc, slots)
    assert werr == 0
    od = op = None
    if attention and w.num_decode:
        nd = w.num_decode
        if w.kv_fp8:
            q64 = w.q_decode.double().numpy()  # bf16 widened exactly
            od = oracle.decode(q64, oracle.dequant_e4m3(kc, w.k_scale), oracle.dequant_e4m3(vc, w.v_scale), bt[:nd],
                               w.context_lens.numpy()[:nd], w.scale, num_threads=threads)
        else:
            od = oracle.decode(storage_numpy(w.q_decode), kc, vc, bt[:nd], w.context_lens.numpy()[:nd], w.scale,
                               num_threads=threads)
    if attention and w.num_chunks:
        op = oracle.prefill(storage_numpy(w.q_prefill), w.cu_q_lens.numpy(), w.q_start_pos.numpy(),
                            w.seq_of_chunk.numpy(), kc, vc, bt, w.context_lens.numpy(), w.scale, num_threads=threads)
    return Expected(slots, err, kc, vc, od, op)
