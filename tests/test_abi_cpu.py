"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_313_gb300 import build as pa_build
from paged_kv_cache_313_gb300 import pa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.lib()


def _declared():
    text = open(HEADER).read()
    return set(re.findall(r"^PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text, flags=re.M))


def test_header_declares_binding_symbols():
    assert _declared() == set(pa.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # nothing else in the pa_ namespace is exported
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.split() and ln.split()[-1].startswith("pa_")}
    assert exported == _declared()


def test_version_and_status_strings(lib):
    assert lib.pa_version() >= 100
    assert lib.pa_status_string(0) == b"ok"
    assert b"workspace" in lib.pa_status_string(pa.PA_ERR_WORKSPACE)
    assert lib.pa_status_string(99) == b"unknown status"


def test_host_side_rejections_need_no_device(lib):
    # invalid sizes are rejected before any CUDA call
    assert lib.pa_slot_mapping(None, 1, 1, None, None, -1, 16, 4, None, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_slot_mapping(None, 1, 1, None, None, 0, 16, 4, None, None, None) == pa.PA_OK  # empty no-op
    assert lib.pa_slot_mapping(None, 1, 1, None, None, 4, 16, 4, None, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv(None, None, 1, 8, 128, 7, None, None, 10, 16, None, None, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_write_kv(None, None, 0, 8, 128, pa.PA_BF16, None, None, 10, 16, None, None, None) == pa.PA_OK
    # head_dim 96 is not built; group 3 heads on 2 kv heads is inconsistent
    args = [None, None, 1, 8, 8, 96, pa.PA_BF16, None, None, 1, 16, None, 1, None, 16, ctypes.c_float(1.0), None, 0,
            None, None]
    assert lib.pa_decode(*args) == pa.PA_ERR_UNSUPPORTED
    args[3], args[4], args[5] = 3, 2, 128
    assert lib.pa_decode(*args) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_workspace_size(4, 3, 2, 128, 16, 100) == 0
    assert lib.pa_decode_plan(-1, 8, 8, 128, 16, 100, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_plan(4, 3, 2, 128, 16, 100, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_plan(4, 8, 8, 96, 16, 100, None, None) == pa.PA_ERR_UNSUPPORTED
    # cascade decode is bf16 only, and takes the decode kernel's head sizes only
    cas = [None, None, 4, 32, 8, 128, pa.PA_F32, None, None, 10, 16, None, 4, None, 100, None, 1, 4, None,
           ctypes.c_float(1.0), None, 0, None, None]
    assert lib.pa_decode_cascade(*cas) == pa.PA_ERR_UNSUPPORTED
    cas[5], cas[6] = 96, pa.PA_BF16
    assert lib.pa_decode_cascade(*cas) == pa.PA_ERR_UNSUPPORTED
    # the no-alloc decode takes exactly the shapes pa_decode takes (one shared check)
    na = [None, None, 1, 8, 8, 96, pa.PA_BF16, None, None, 1, 16, None, 1, None, 16, ctypes.c_float(1.0), None, None]
    assert lib.pa_decode_noalloc(*na) == pa.PA_ERR_UNSUPPORTED
    na[3], na[4], na[5] = 3, 2, 128
    assert lib.pa_decode_noalloc(*na) == pa.PA_ERR_INVALID_ARG
    na[3], na[4], na[10] = 8, 8, 2048
    assert lib.pa_decode_noalloc(*na) == pa.PA_ERR_UNSUPPORTED
    args[3], args[4], args[10] = 8, 8, 2048
    assert lib.pa_decode(*args) == pa.PA_ERR_UNSUPPORTED
    # the bounded-wait self-check: poll limit and result pointer are checked on the host
    assert lib.pa_check_bounded_wait(0, 0, ctypes.c_void_p(16), None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_check_bounded_wait(1 << 17, 0, ctypes.c_void_p(16), None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_check_bounded_wait(100, 0, None, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(None, None, 4, 16, 8, 128, pa.PA_BF16, None, None, None, 0, None, None) == pa.PA_OK
    assert lib.pa_copy_blocks(None, None, 4, 16, 8, 128, pa.PA_BF16, None, None, None, 2, None, None) == \
        pa.PA_ERR_INVALID_ARG


def test_binding_raises_without_cuda_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        pa.pa_slot_mapping(torch.zeros(1, 1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                           torch.zeros(1, dtype=torch.int32), 16, 4, slot_mapping=torch.zeros(1, dtype=torch.int64))
