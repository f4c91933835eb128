"""pa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory where decode runs (a runtime that forbids allocation after
start-up, a plugin inside another framework's memory budget, code that must
not trigger the synchronisation an allocation can cause).  It takes its
split-KV scratch from the library's fixed 16 MiB device array instead of a
caller workspace.

Checked through the C ABI against the fp64 oracle at the stated tolerances
(1e-5 fp32, 2e-2 bf16), on two calls in a row: the array keeps the previous
call's contents, so the second call shows that what must start at zero is
cleared.  One batch needs more than 16 MiB of scratch under pa_decode's own
plan, so the entry point must lengthen its partitions to fit; it is also
compared with pa_decode on that batch.

Named so that pytest collects it last: a run that stops at the first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_313_gb300 import pa
from paged_kv_cache_313_gb300 import workloads as W
from paged_kv_cache_313_gb300.runner import DeviceStep
from paged_kv_cache_313_gb300.workloads import storage_numpy

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}
SCRATCH_BYTES = 16 << 20


def _maxabs(got: torch.Tensor, want: np.ndarray) -> float:
    g = got.float().cpu().double().numpy()
    assert np.all(np.isfinite(g))
    return float(np.max(np.abs(g - want)))


def _twice(args, want, tol):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full(want.shape, float("nan"), dtype=args[0].dtype, device="cuda")
        pa.pa_decode_noalloc(*args, out=out, error_count=err)
        torch.cuda.synchronize()
        diff = _maxabs(out, want)
        assert diff <= tol, diff
    assert int(err.item()) == 0
    return out


@pytest.mark.parametrize("name", ["tiny_fp32", "decode_bf16"])
def test_noalloc_matches_oracle_twice(name):
    w = W.tiny_fp32(0) if name == "tiny_fp32" else W.small("decode_bf16", 0)
    st = DeviceStep(w)
    st.slot_mapping()
    st.write_kv()
    torch.cuda.synchronize()
    nd = w.num_decode
    kc, vc = storage_numpy(st.k_cache.cpu()), storage_numpy(st.v_cache.cpu())
    want = oracle.decode(storage_numpy(w.q_decode), kc, vc, w.block_tables.numpy()[:nd],
                         w.context_lens.numpy()[:nd], w.scale)
    args = (st.q_decode, st.k_cache, st.v_cache, st.block_tables[:nd], st.context_lens[:nd], st.max_context_len,
            w.scale)
    _twice(args, want, TOL[w.dtype])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_lengthens_partitions_to_fit_its_scratch(dtype):
    """512 sequences of one kv head with 8 query heads and contexts up to 8192 tokens: pa_decode's plan
    (768-token partitions) needs more scratch, more than the 16 MiB array holds, so
    this call succeeds only with longer partitions (pa_decode's plan also reserves room for the quarter-length partitions of the batch's last sequences).  Block tables draw their entries from a pool of 700 blocks
    (a block may appear in several tables), which keeps the pool small."""
    rng = np.random.default_rng(31)
    N, Hq, Hkv, D, B, P, max_ctx = 512, 8, 1, 128, 16, 700, 8192
    need = pa.pa_decode_workspace_size(N, Hq, Hkv, D, B, max_ctx)
    assert need > SCRATCH_BYTES, need
    part, splits = pa.pa_decode_plan(N, Hq, Hkv, D, B, max_ctx)
    assert splits > 1
    lens = rng.integers(1, 1500, size=N).astype(np.int32)
    lens[rng.choice(N, 24, replace=False)] = rng.integers(4000, max_ctx + 1, size=24)
    lens[7] = max_ctx
    width = max_ctx // B
    tables = rng.integers(0, P, size=(N, width)).astype(np.int32)
    kc = rng.standard_normal((P, B, Hkv, D), dtype=np.float32)
    vc = rng.standard_normal((P, B, Hkv, D), dtype=np.float32)
    q = rng.standard_normal((N, Hq, D), dtype=np.float32)
    scale = 1 / np.sqrt(D)
    t = lambda x: torch.from_numpy(x).to(dtype).cuda()  # noqa: E731
    qd, kd, vd = t(q), t(kc), t(vc)
    st = lambda x: storage_numpy(x.cpu())  # noqa: E731
    want = oracle.decode(st(qd), st(kd), st(vd), tables, lens, scale)
    bt, ctx = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    got = _twice((qd, kd, vd, bt, ctx, max_ctx, scale), want, TOL[dtype])
    # pa_decode on the same inputs (its own plan and a caller workspace) agrees within the same bound
    ws = pa.new_decode_workspace(N, Hq, Hkv, D, B, max_ctx)
    ref = pa.pa_decode(qd, kd, vd, bt, ctx, max_ctx, scale, ws)
    torch.cuda.synchronize()
    assert _maxabs(ref, want) <= TOL[dtype]
    assert float((got.float() - ref.float()).abs().max()) <= TOL[dtype]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = W.small("decode_bf16", 0)
    st = DeviceStep(w)
    # a batch whose split-KV scratch exceeds 16 MiB even with one partition per sequence
    big_n = 4096
    q = torch.zeros(big_n, w.num_q_heads, w.head_dim, dtype=w.dtype, device="cuda")
    bt = st.block_tables[:1].repeat(big_n, 1)
    ctx = st.context_lens[:1].repeat(big_n)
    need = pa.pa_decode_workspace_size(big_n, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, 32768)
    assert need > SCRATCH_BYTES
    with pytest.raises(pa.PaError) as ei:
        pa.pa_decode_noalloc(q, st.k_cache, st.v_cache, bt, ctx, 32768, w.scale)
    assert ei.value.status == pa.PA_ERR_WORKSPACE
