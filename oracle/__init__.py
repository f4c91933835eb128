"""Plain fp64 CPU oracle for the paged-attention hot path.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The oracle is plain C
(``pa_oracle.c``) behind this ctypes wrapper; it shares no code with the CUDA
library and never imports the package.

Inputs are numpy arrays.  Floating-point tensors are passed in their storage
form: ``np.float32`` for fp32, ``np.uint16`` holding the bf16 bit patterns for
bf16 (numpy has no bf16 type).  Outputs of the attention routines are fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

F32 = 0
BF16 = 1
F64 = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no tuning) and return the path."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32p, i64p, vp, dp = (ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p,
                                       ctypes.POINTER(ctypes.c_double))
            lib.oracle_num_blocks.argtypes = [i64, i64]
            lib.oracle_num_blocks.restype = i64
            lib.oracle_slot_mapping.argtypes = [i32p, i64, i64, i32p, i32p, i64, i64, i64, i64p]
            lib.oracle_map_to_kernel_blocks.argtypes = [i32p, i64, i64, i64, i32p, i64]
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_write_kv_fp8.argtypes = [vp, vp, i64, i64, i64, vp, vp, i64, i64, i64p, ctypes.c_float,
                                                ctypes.c_float]
            lib.oracle_dequant_e4m3.argtypes = [vp, i64, ctypes.c_float, dp]
            lib.oracle_dequant_e4m3.restype = None
            lib.oracle_map_to_kernel_blocks.restype = None
            lib.oracle_slot_mapping.restype = ctypes.c_int
            lib.oracle_write_kv.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int, vp, vp, i64, i64, i64p]
            lib.oracle_write_kv.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [dp, vp, i64, i64, i64, i64, ctypes.c_int, vp, vp, i64, i64,
                                          i32p, i64, i32p, ctypes.c_double, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_prefill.argtypes = [dp, vp, i32p, i32p, i32p, i64, i64, i64, i64, i64, ctypes.c_int,
                                           vp, vp, i64, i64, i32p, i64, i32p, ctypes.c_double, ctypes.c_int]
            lib.oracle_prefill.restype = ctypes.c_int
            _lib = lib
    return _lib


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle storage dtype must be float32, float64 or uint16 (bf16 bits), got {a.dtype}")


def _threads(num_threads):
    return num_threads if num_threads else (os.cpu_count() or 1)


def num_blocks(seq_len: int, block_size: int) -> int:
    """ceil(seq_len / block_size); 0 for an empty sequence."""
    return int(_load().oracle_num_blocks(int(seq_len), int(block_size)))


def slot_mapping(block_tables, seq_idx, pos, block_size: int, num_blocks: int):
    """Slots of the new tokens (int64, -1 for padding/invalid) and the error count."""
    bt, btp = _i32(block_tables)
    si, sip = _i32(seq_idx)
    ps, psp = _i32(pos)
    out = np.empty(si.shape[0], dtype=np.int64)
    rc = _load().oracle_slot_mapping(btp, bt.shape[0], bt.shape[1], sip, psp, si.shape[0], block_size,
                                     num_blocks, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    return out, -rc


def map_to_kernel_blocks(mgr_tables, ratio: int, kernel_width: int | None = None):
    """Kernel-side block tables for manager blocks of ratio kernel blocks each."""
    mt, mtp = _i32(mgr_tables)
    S, W = mt.shape
    kw = W * ratio if kernel_width is None else int(kernel_width)
    out = np.empty((S, kw), dtype=np.int32)
    _load().oracle_map_to_kernel_blocks(mtp, S, W, int(ratio), out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        kw)
    return out


def e4m3_value(code: int) -> float:
    """Value of an e4m3 code (NaN for the NaN codes)."""
    return float(_load().oracle_e4m3_value(int(code)))


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code to float32 x (ties to even, saturating at 448)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def write_kv_fp8(k_new, v_new, k_cache, v_cache, slots, k_scale: float, v_scale: float) -> int:
    """Quantising write into uint8 e4m3 pools, in place: code = e4m3(x * (1/scale)); returns the error count."""
    assert k_cache.dtype == v_cache.dtype == np.uint8 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    T, H, D = k_new.shape
    P, B = k_cache.shape[0], k_cache.shape[1]
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    rc = _load().oracle_write_kv_fp8(k_new.ctypes.data, v_new.ctypes.data, T, H, D, k_cache.ctypes.data,
                                     v_cache.ctypes.data, P, B, sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                     float(k_scale), float(v_scale))
    return -rc


def dequant_e4m3(codes, scale: float) -> np.ndarray:
    """codes * scale in float64 (exact)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_dequant_e4m3(c.ctypes.data, c.size, float(scale), out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def write_kv(k_new, v_new, k_cache, v_cache, slots) -> int:
    """Copy each token's K/V row into the pools at its slot, in place; returns the error count."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    dt = _dtype_code(k_cache)
    assert k_new.dtype == k_cache.dtype == v_new.dtype == v_cache.dtype
    T, H, D = k_new.shape
    P, B = k_cache.shape[0], k_cache.shape[1]
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    rc = _load().oracle_write_kv(k_new.ctypes.data, v_new.ctypes.data, T, H, D, dt, k_cache.ctypes.data,
                                 v_cache.ctypes.data, P, B, sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    return -rc


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, num_threads: int = 0):
    """fp64 decode attention: q [N, Hq, D]; pools [P, B, Hkv, D]; returns [N, Hq, D] fp64."""
    q = np.ascontiguousarray(q)
    dt = _dtype_code(q)
    assert q.dtype == k_cache.dtype == v_cache.dtype
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    assert D2 == D
    bt, btp = _i32(block_tables)
    cl, clp = _i32(context_lens)
    assert bt.shape[0] == N and cl.shape[0] == N
    out = np.zeros((N, Hq, D), dtype=np.float64)
    rc = _load().oracle_decode(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), q.ctypes.data, N, Hq, Hkv, D,
                               dt, np.ascontiguousarray(k_cache).ctypes.data,
                               np.ascontiguousarray(v_cache).ctypes.data, P, B, btp, bt.shape[1], clp,
                               float(scale), _threads(num_threads))
    if rc != 0:
        raise ValueError("oracle.decode: block table or context length out of range")
    return out


def prefill(q, cu_q_lens, q_start_pos, seq_of_chunk, k_cache, v_cache, block_tables, context_lens,
            scale: float, num_threads: int = 0):
    """fp64 causal chunked-prefill attention: q [total_q, Hq, D]; returns [total_q, Hq, D] fp64."""
    q = np.ascontiguousarray(q)
    dt = _dtype_code(q)
    assert q.dtype == k_cache.dtype == v_cache.dtype
    T, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    assert D2 == D
    cu, cup = _i32(cu_q_lens)
    qs, qsp = _i32(q_start_pos)
    sc, scp = _i32(seq_of_chunk)
    bt, btp = _i32(block_tables)
    cl, clp = _i32(context_lens)
    C = qs.shape[0]
    assert cu.shape[0] == C + 1 and int(cu[-1]) == T
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = _load().oracle_prefill(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), q.ctypes.data, cup, qsp, scp,
                                C, bt.shape[0], Hq, Hkv, D, dt, np.ascontiguousarray(k_cache).ctypes.data,
                                np.ascontiguousarray(v_cache).ctypes.data, P, B, btp, bt.shape[1], clp,
                                float(scale), _threads(num_threads))
    if rc != 0:
        raise ValueError("oracle.prefill: chunk, block table or context length out of range")
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
