"""pa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (it uses the library's fixed 16 MiB device scratch array instead
of a caller workspace).  Checked through the C ABI against pa_decode on the
same inputs, on two calls in a row (the array keeps the previous call's
contents, so the second call shows that what must start at zero is cleared).

Named so that pytest collects it last: a run that stops at the first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_313_gb300 import pa
from paged_kv_cache_313_gb300 import workloads as W
from paged_kv_cache_313_gb300.runner import DeviceStep

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


@pytest.mark.parametrize("name", ["tiny_fp32", "decode_bf16"])
def test_noalloc_matches_pa_decode_twice(name):
    w = W.tiny_fp32(0) if name == "tiny_fp32" else W.small("decode_bf16", 0)
    st = DeviceStep(w)
    st.slot_mapping()
    st.write_kv()
    want = st.decode().clone()
    nd = w.num_decode
    args = (st.q_decode, st.k_cache, st.v_cache, st.block_tables[:nd], st.context_lens[:nd], st.max_context_len,
            w.scale)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full_like(want, float("nan"))
        pa.pa_decode_noalloc(*args, out=out, error_count=err)
        torch.cuda.synchronize()
        diff = (out.double() - want.double()).abs().max().item()
        assert np.isfinite(diff) and diff <= TOL[w.dtype], diff
    assert int(err.item()) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = W.small("decode_bf16", 0)
    st = DeviceStep(w)
    nd = w.num_decode
    # a batch whose split-KV scratch would exceed 16 MiB: many sequences, long maximum context
    big_n = 4096
    q = torch.zeros(big_n, w.num_q_heads, w.head_dim, dtype=w.dtype, device="cuda")
    bt = st.block_tables[:1].repeat(big_n, 1)
    ctx = st.context_lens[:1].repeat(big_n)
    need = pa.pa_decode_workspace_size(big_n, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, 32768)
    assert need > (16 << 20)
    with pytest.raises(pa.PaError) as ei:
        pa.pa_decode_noalloc(q, st.k_cache, st.v_cache, bt, ctx, 32768, w.scale)
    assert ei.value.status == pa.PA_ERR_WORKSPACE
    del nd
