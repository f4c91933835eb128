"""Python binding of libpa.so: the C ABI in include/pa.h, same names, torch
CUDA tensors in and out.  Argument marshalling only — every step runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_WORKSPACE, PA_ERR_UNSUPPORTED_DEVICE = range(6)
PA_F32, PA_BF16 = 0, 1

# Every symbol include/pa.h declares.
SYMBOLS = ("pa_version", "pa_status_string", "pa_last_cuda_error", "pa_slot_mapping", "pa_write_kv",
           "pa_write_kv_paged", "pa_write_kv_paged_fp8", "pa_decode_workspace_size", "pa_decode_plan", "pa_decode", "pa_decode_fp8", "pa_decode_write",
           "pa_decode_write_fp8",
           "pa_decode_cascade_workspace_size", "pa_decode_cascade", "pa_decode_noalloc", "pa_prefill_workspace_size",
           "pa_prefill_chunk", "pa_copy_blocks", "pa_map_to_kernel_blocks", "pa_stage_copy",
           "pa_check_bounded_wait")


class PaError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str, cuda_error: int = 0):
        super().__init__(f"{fn}: {message} (status {status}" + (f", cudaError {cuda_error})" if cuda_error else ")"))
        self.status = status
        self.cuda_error = cuda_error


_lock = threading.Lock()
_lib = None

_i, _sz, _p, _f = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
_SIGNATURES = {
    "pa_version": ([], _i),
    "pa_status_string": ([_i], ctypes.c_char_p),
    "pa_last_cuda_error": ([], _i),
    "pa_slot_mapping": ([_p, _i, _i, _p, _p, _i, _i, _i, _p, _p, _p], _i),
    "pa_write_kv": ([_p, _p, _i, _i, _i, _i, _p, _p, _i, _i, _p, _p, _p], _i),
    "pa_write_kv_paged": ([_p, _p, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _i, _p, _p, _p, _p, _p], _i),
    "pa_write_kv_paged_fp8": ([_p, _p, _i, _i, _i, _p, _p, _i, _i, _p, _i, _i, _p, _p, _p, _f, _f, _p, _p], _i),
    "pa_decode_workspace_size": ([_i, _i, _i, _i, _i, _i], _sz),
    "pa_decode_plan": ([_i, _i, _i, _i, _i, _i, _p, _p], _i),
    "pa_decode": ([_p, _p, _i, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _f, _p, _sz, _p, _p], _i),
    "pa_decode_fp8": ([_p, _p, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _f, _f, _f, _p, _sz, _p, _p], _i),
    "pa_decode_write_fp8": ([_p, _p, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _f, _f, _f, _p, _p, _p, _p, _sz,
                             _p, _p], _i),
    "pa_decode_write": ([_p, _p, _i, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _f, _p, _p, _p, _p, _sz, _p,
                         _p], _i),
    "pa_decode_cascade_workspace_size": ([_i, _i, _i, _i, _i, _i], _sz),
    "pa_decode_cascade": ([_p, _p, _i, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _p, _i, _i, _p, _f, _p, _sz,
                           _p, _p], _i),
    "pa_decode_noalloc": ([_p, _p, _i, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _f, _p, _p], _i),
    "pa_prefill_workspace_size": ([_i, _i, _i, _i, _i, _i], _sz),
    "pa_prefill_chunk": ([_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _f, _p,
                          _sz, _p, _p], _i),
    "pa_stage_copy": ([_p, _p, _sz, _p], _i),
    "pa_check_bounded_wait": ([_i, _i, _p, _p, _p], _i),
    "pa_map_to_kernel_blocks": ([_p, _i, _i, _i, _p, _i, _p], _i),
    "pa_copy_blocks": ([_p, _p, _i, _i, _i, _i, _i, _p, _p, _p, _i, _p, _p], _i),
}


def lib() -> ctypes.CDLL:
    """The loaded libpa.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run "
                                   "`python -m paged_kv_cache_313_gb300.build` first")
            h = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(h, name)
                fn.argtypes = args
                fn.restype = res
            _lib = h
    return _lib


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        L = lib()
        raise PaError(fn, status, L.pa_status_string(status).decode(),
                      L.pa_last_cuda_error() if status == PA_ERR_CUDA else 0)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev(t: torch.Tensor | None, name: str, dtype=None, host_ok: bool = False):
    """Pointer of a contiguous CUDA tensor (or, with host_ok, of a pinned host tensor, which the device reaches
    through its mapping)."""
    if t is None:
        return None
    if not (t.is_cuda or (host_ok and t.is_pinned())):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pa_version() -> int:
    return lib().pa_version()


def pa_slot_mapping(block_tables, seq_idx, pos, block_size: int, num_blocks: int, slot_mapping=None,
                    error_count=None, stream=None) -> torch.Tensor:
    """slot = block_tables[seq, pos // B] * B + pos % B for each new token (int64, -1 = skip)."""
    T = seq_idx.numel()
    if slot_mapping is None:
        slot_mapping = torch.empty(T, dtype=torch.int64, device=seq_idx.device)
    S, W = block_tables.shape
    _check("pa_slot_mapping", lib().pa_slot_mapping(
        _dev(block_tables, "block_tables", torch.int32), S, W, _dev(seq_idx, "seq_idx", torch.int32),
        _dev(pos, "pos", torch.int32), T, int(block_size), int(num_blocks),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(error_count, "error_count", torch.int32),
        _stream(stream)))
    return slot_mapping


def pa_write_kv(k_new, v_new, k_cache, v_cache, slot_mapping, error_count=None, stream=None) -> None:
    """Scatter each new token's K/V row into the pools at its slot (bit-exact)."""
    T, H, D = k_new.shape
    P, B = k_cache.shape[0], k_cache.shape[1]
    dt = _dtype_code(k_new)
    for name, t in (("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != k_new.dtype:
            raise TypeError(f"{name} dtype {t.dtype} differs from k_new {k_new.dtype}")
    _check("pa_write_kv", lib().pa_write_kv(
        _dev(k_new, "k_new"), _dev(v_new, "v_new"), T, H, D, dt, _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        P, B, _dev(slot_mapping, "slot_mapping", torch.int64), _dev(error_count, "error_count", torch.int32),
        _stream(stream)))


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len) -> int:
    return int(lib().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                              max_context_len))


def pa_write_kv_paged(k_new, v_new, k_cache, v_cache, block_tables, seq_idx, pos, slot_mapping=None,
                      error_count=None, stream=None):
    """Slot mapping and K/V scatter in one launch (bit-exact); slot_mapping, if given, receives the slots."""
    T, H, D = k_new.shape
    P, B = k_cache.shape[0], k_cache.shape[1]
    S, W = block_tables.shape
    for name, t in (("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != k_new.dtype:
            raise TypeError(f"{name} dtype {t.dtype} differs from k_new {k_new.dtype}")
    _check("pa_write_kv_paged", lib().pa_write_kv_paged(
        _dev(k_new, "k_new"), _dev(v_new, "v_new"), T, H, D, _dtype_code(k_new), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), P, B, _dev(block_tables, "block_tables", torch.int32), S, W,
        _dev(seq_idx, "seq_idx", torch.int32), _dev(pos, "pos", torch.int32),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(error_count, "error_count", torch.int32),
        _stream(stream)))
    return slot_mapping


def pa_write_kv_paged_fp8(k_new, v_new, k_cache, v_cache, block_tables, seq_idx, pos, k_scale: float,
                          v_scale: float, slot_mapping=None, error_count=None, stream=None):
    """Slot mapping and a quantising K/V write into uint8 e4m3 pools (code = e4m3(x / scale))."""
    T, H, D = k_new.shape
    P, B = k_cache.shape[0], k_cache.shape[1]
    S, W = block_tables.shape
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("fp8 pools are uint8 tensors of e4m3 codes")
    _check("pa_write_kv_paged_fp8", lib().pa_write_kv_paged_fp8(
        _dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16), T, H, D,
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), P, B, _dev(block_tables, "block_tables", torch.int32),
        S, W, _dev(seq_idx, "seq_idx", torch.int32), _dev(pos, "pos", torch.int32),
        _dev(slot_mapping, "slot_mapping", torch.int64), float(k_scale), float(v_scale),
        _dev(error_count, "error_count", torch.int32), _stream(stream)))
    return slot_mapping


def pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len):
    """(partition length in tokens, number of partitions) pa_decode uses for these sizes."""
    part, splits = ctypes.c_int(0), ctypes.c_int(0)
    _check("pa_decode_plan", lib().pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                                  max_context_len, ctypes.byref(part), ctypes.byref(splits)))
    return part.value, splits.value


def new_decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                         device=None) -> torch.Tensor:
    """A zeroed workspace of the size pa_decode needs (reusable across calls on one stream)."""
    n = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len)
    if n == 0:
        raise PaError("pa_decode_workspace_size", PA_ERR_UNSUPPORTED, "unsupported sizes or device")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float, workspace,
              out=None, error_count=None, stream=None) -> torch.Tensor:
    """Paged decode attention: out[s, h] = softmax(scale q[s,h] K_s^T) V_s over context_lens[s] tokens."""
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_cache differ")
    if out is None:
        out = torch.empty_like(q)
    _check("pa_decode", lib().pa_decode(
        _dev(out, "out", q.dtype, host_ok=True),
        _dev(q, "q"), N, Hq, Hkv, D, _dtype_code(q), _dev(k_cache, "k_cache", q.dtype),
        _dev(v_cache, "v_cache", q.dtype), P, B, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(error_count, "error_count", torch.int32), _stream(stream)))
    return out


def pa_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                  k_scale: float, v_scale: float, workspace, out=None, error_count=None, stream=None) -> torch.Tensor:
    """pa_decode over uint8 e4m3 pools read back as code * scale; q and out bf16."""
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_cache differ")
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("fp8 pools are uint8 tensors of e4m3 codes")
    if out is None:
        out = torch.empty_like(q)
    _check("pa_decode_fp8", lib().pa_decode_fp8(
        _dev(out, "out", torch.bfloat16, host_ok=True),
        _dev(q, "q", torch.bfloat16), N, Hq, Hkv, D, _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), P, B, _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale), float(k_scale),
        float(v_scale), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(error_count, "error_count", torch.int32), _stream(stream)))
    return out


def pa_decode_write_fp8(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                        k_scale: float, v_scale: float, k_new, v_new, workspace, out=None, new_slots=None,
                        error_count=None, stream=None) -> torch.Tensor:
    """pa_decode_fp8 that also stores each sequence's newest token (bf16 K/V rows k_new/v_new [N, Hkv, D]) into the
    e4m3 pools at its slot, quantised as e4m3(x * (1/scale)), in the same launch."""
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(k_new.shape) != (N, Hkv, D) or tuple(v_new.shape) != (N, Hkv, D):
        raise ValueError("shapes of q, k_cache, k_new, v_new disagree")
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("fp8 pools are uint8 tensors of e4m3 codes")
    if out is None:
        out = torch.empty_like(q)
    _check("pa_decode_write_fp8", lib().pa_decode_write_fp8(
        _dev(out, "out", torch.bfloat16, host_ok=True),
        _dev(q, "q", torch.bfloat16), N, Hq, Hkv, D, _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), P, B,
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale), float(k_scale),
        float(v_scale), _dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16),
        _dev(new_slots, "new_slots", torch.int64), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev(error_count, "error_count", torch.int32),
        _stream(stream)))
    return out


def pa_decode_write(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float, k_new,
                    v_new, workspace, out=None, new_slots=None, error_count=None, stream=None) -> torch.Tensor:
    """pa_decode that also writes each sequence's newest token (K/V rows k_new/v_new [N, Hkv, D]) into the
    pools at its slot, in the same launch."""
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(k_new.shape) != (N, Hkv, D) or tuple(v_new.shape) != (N, Hkv, D):
        raise ValueError("shapes of q, k_cache, k_new, v_new disagree")
    if out is None:
        out = torch.empty_like(q)
    _check("pa_decode_write", lib().pa_decode_write(
        _dev(out, "out", q.dtype, host_ok=True),
        _dev(q, "q"), N, Hq, Hkv, D, _dtype_code(q), _dev(k_cache, "k_cache", q.dtype),
        _dev(v_cache, "v_cache", q.dtype), P, B, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        _dev(k_new, "k_new", q.dtype), _dev(v_new, "v_new", q.dtype), _dev(new_slots, "new_slots", torch.int64),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(error_count, "error_count", torch.int32), _stream(stream)))
    return out


def new_cascade_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                          device=None) -> torch.Tensor:
    """A zeroed workspace of the size pa_decode_cascade needs."""
    n = int(lib().pa_decode_cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                                   max_context_len))
    if n == 0:
        raise PaError("pa_decode_cascade_workspace_size", PA_ERR_UNSUPPORTED, "unsupported sizes or device")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode_cascade(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, group_offsets,
                      max_group_size: int, prefix_lens, scale: float, workspace, out=None, error_count=None,
                      stream=None) -> torch.Tensor:
    """pa_decode where each group of sequences [group_offsets[g], group_offsets[g+1]) shares its first
    prefix_lens[s] context tokens: the shared prefix is read once per group (bf16, head_dim 128)."""
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_cache differ")
    if out is None:
        out = torch.empty_like(q)
    G = group_offsets.numel() - 1
    _check("pa_decode_cascade", lib().pa_decode_cascade(
        _dev(out, "out", q.dtype, host_ok=True),
        _dev(q, "q"), N, Hq, Hkv, D, _dtype_code(q), _dev(k_cache, "k_cache", q.dtype),
        _dev(v_cache, "v_cache", q.dtype), P, B, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len),
        _dev(group_offsets, "group_offsets", torch.int32), G, int(max_group_size),
        _dev(prefix_lens, "prefix_lens", torch.int32), float(scale), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev(error_count, "error_count", torch.int32),
        _stream(stream)))
    return out


def pa_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                      out=None, error_count=None, stream=None) -> torch.Tensor:
    """pa_decode without a workspace argument, for callers that cannot allocate
    device memory: the split-KV scratch is the library's own fixed 16 MiB device
    array.  Sizes that need more scratch raise PaError (PA_ERR_WORKSPACE).
    Calls that may overlap on the GPU share that array and race."""
    N, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_cache differ")
    if out is None:
        out = torch.empty_like(q)
    _check("pa_decode_noalloc", lib().pa_decode_noalloc(
        _dev(out, "out", q.dtype, host_ok=True),
        _dev(q, "q"), N, Hq, Hkv, D, _dtype_code(q), _dev(k_cache, "k_cache", q.dtype),
        _dev(v_cache, "v_cache", q.dtype), P, B, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        _dev(error_count, "error_count", torch.int32), _stream(stream)))
    return out


def pa_prefill_workspace_size(num_chunks, max_q_len, num_q_heads, num_kv_heads, head_dim, block_size) -> int:
    return int(lib().pa_prefill_workspace_size(num_chunks, max_q_len, num_q_heads, num_kv_heads, head_dim,
                                               block_size))


def pa_prefill_chunk(q, cu_q_lens, q_start_pos, seq_of_chunk, max_q_len: int, k_cache, v_cache, block_tables,
                     context_lens, scale: float, workspace=None, out=None, error_count=None,
                     stream=None) -> torch.Tensor:
    """Causal chunked-prefill attention over the paged pool."""
    T, Hq, D = q.shape
    P, B, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_cache differ")
    if out is None:
        out = torch.empty_like(q)
    C = q_start_pos.numel()
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pa_prefill_chunk", lib().pa_prefill_chunk(
        _dev(out, "out", q.dtype, host_ok=True), _dev(q, "q"), _dev(cu_q_lens, "cu_q_lens", torch.int32),
        _dev(q_start_pos, "q_start_pos", torch.int32), _dev(seq_of_chunk, "seq_of_chunk", torch.int32), C, T,
        int(max_q_len), block_tables.shape[0], Hq, Hkv, D, _dtype_code(q), _dev(k_cache, "k_cache", q.dtype),
        _dev(v_cache, "v_cache", q.dtype), P, B, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), float(scale), ws_ptr, ws_bytes,
        _dev(error_count, "error_count", torch.int32), _stream(stream)))
    return out


def pa_copy_blocks(k_cache, v_cache, src_blocks, dst_blocks, num_valid, error_count=None, stream=None) -> None:
    """Copy-on-write: copy the first num_valid[i] slots of block src_blocks[i] into dst_blocks[i]."""
    P, B, H, D = k_cache.shape
    _check("pa_copy_blocks", lib().pa_copy_blocks(
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache", k_cache.dtype), P, B, H, D, _dtype_code(k_cache),
        _dev(src_blocks, "src_blocks", torch.int32), _dev(dst_blocks, "dst_blocks", torch.int32),
        _dev(num_valid, "num_valid", torch.int32), src_blocks.numel(), _dev(error_count, "error_count", torch.int32),
        _stream(stream)))


def pa_stage_copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy src into dst (same number of bytes) with a kernel; either may be a pinned host tensor."""
    for name, t in (("dst", dst), ("src", src)):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("dst and src sizes differ")
    _check("pa_stage_copy", lib().pa_stage_copy(dst.data_ptr(), src.data_ptr(), n, _stream(stream)))
    return dst


def pa_map_to_kernel_blocks(mgr_tables, ratio: int, kernel_tables=None, stream=None) -> torch.Tensor:
    """Kernel block tables for manager blocks of `ratio` kernel blocks: entry j of row s is
    mgr_tables[s, j // ratio] * ratio + j % ratio (-1 for -1)."""
    S, W = mgr_tables.shape
    if kernel_tables is None:
        kernel_tables = torch.empty(S, W * ratio, dtype=torch.int32, device=mgr_tables.device)
    _check("pa_map_to_kernel_blocks", lib().pa_map_to_kernel_blocks(
        _dev(mgr_tables, "mgr_tables", torch.int32), S, W, int(ratio),
        _dev(kernel_tables, "kernel_tables", torch.int32), kernel_tables.shape[1], _stream(stream)))
    return kernel_tables


def pa_check_bounded_wait(polls: int, arrive: bool, device="cuda", stream=None):
    """Run the library's bounded-wait self-check: one warp waits `polls` polls on an mbarrier that nothing
    arrives on (arrive=False) or that it arrived on first.  Returns (result, errors) after synchronising:
    result 1 if the wait succeeded, 0 if it gave up; errors the count it added."""
    result = torch.full((1,), -1, dtype=torch.int32, device=device)
    errors = torch.zeros(1, dtype=torch.int32, device=device)
    _check("pa_check_bounded_wait", lib().pa_check_bounded_wait(int(polls), 1 if arrive else 0,
                                                                _dev(result, "result", torch.int32),
                                                                _dev(errors, "error_count", torch.int32),
                                                                _stream(stream)))
    torch.cuda.synchronize(result.device)
    return int(result.item()), int(errors.item())
