"""GPU parity of the hot path against the CPU oracle, through the C ABI.

Bit-exact: slot mapping, KV write (whole pools compared), copy-on-write copy.
Attention: max-abs error against the fp64 oracle, 1e-5 for fp32 and 2e-2 for
bf16 workloads.  Reduced workloads span several partitions, tiles and ragged
tails; the full workloads are the ones the benchmark times, in the same
launch configuration.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_313_gb300 import pa
from paged_kv_cache_313_gb300 import workloads as W
from paged_kv_cache_313_gb300.allocator import BlockAllocator
from paged_kv_cache_313_gb300.runner import DeviceStep
from paged_kv_cache_313_gb300.workloads import storage_numpy

from oracle_step import expected_step

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}

_cache = {}


def _case(kind, name):
    key = (kind, name)
    if key not in _cache:
        w = W.make(name, 0) if kind == "full" else W.small(name, 0)
        _cache.clear()  # keep one large workload resident at a time
        _cache[key] = (w, expected_step(w))
    return _cache[key]


CASES = [("small", n) for n in ("tiny_fp32", "decode_bf16", "longctx_bf16", "shared_prefix_bf16", "mixed_bf16",
                                 "decode_fp8")] + \
        [("full", n) for n in ("decode_bf16", "longctx_bf16", "shared_prefix_bf16", "shared_prefix_cow_bf16",
                               "mixed_bf16", "decode_fp8")]


def _maxabs(got: torch.Tensor, want: np.ndarray) -> float:
    g = got.float().cpu().double().numpy()
    assert np.all(np.isfinite(g))
    return float(np.max(np.abs(g - want))) if want.size else 0.0


@pytest.mark.parametrize("kind,name", CASES)
def test_step_parity(kind, name):
    w, exp = _case(kind, name)
    st = DeviceStep(w)
    if w.kv_fp8:
        st.write_kv_paged()  # the quantising write maps the slots itself and records them
    else:
        st.slot_mapping()
    assert torch.equal(st.slots.cpu(), torch.from_numpy(exp.slots)), "slot mapping differs"
    if not w.kv_fp8:
        st.write_kv()
    kc = storage_numpy(st.k_cache.cpu())
    vc = storage_numpy(st.v_cache.cpu())
    assert np.array_equal(kc, exp.k_cache) and np.array_equal(vc, exp.v_cache), "pool contents differ after write"
    out_d = st.decode()
    if w.num_decode:
        err = _maxabs(out_d, exp.out_decode)
        assert err <= TOL[w.dtype], f"decode max-abs error {err}"
    if w.num_chunks:
        out_p = st.prefill()
        err = _maxabs(out_p, exp.out_prefill)
        assert err <= TOL[w.dtype], f"prefill max-abs error {err}"
    torch.cuda.synchronize()
    assert st.errors() == 0


@pytest.mark.parametrize("name", ["decode_bf16", "mixed_bf16"])
def test_repeat_runs_bitwise_identical(name):
    w, _ = _case("small", name)
    st = DeviceStep(w)
    a = [t.clone() for t in st.run()]
    for _ in range(3):
        b = st.run()
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_slot_mapping_invalid_entries_match_oracle():
    bt = np.array([[3, -1], [0, 1]], dtype=np.int32)
    seq = np.array([0, 0, 1, 1, 0, 2, -1, 1], np.int32)
    pos = np.array([5, -1, 9, 20, 17, 0, 0, 40], np.int32)
    want, nerr = oracle.slot_mapping(bt, seq, pos, 16, 4)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pa.pa_slot_mapping(torch.from_numpy(bt).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                             16, 4, error_count=err)
    assert got.cpu().tolist() == want.tolist()
    assert int(err.item()) == nerr == 4


def test_write_kv_skips_padding_and_rejects_out_of_pool():
    kc = torch.zeros(2, 4, 2, 8, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones(3, 2, 8, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv(kn, 2 * kn, kc, vc, torch.tensor([-1, 5, 8], device="cuda"), error_count=err)
    assert int(err.item()) == 1
    assert torch.count_nonzero(kc).item() == 16 and torch.all(kc.view(8, 16)[5] == 1)
    assert torch.all(vc.view(8, 16)[5] == 2)


def test_copy_blocks_matches_host_copy():
    g = torch.Generator().manual_seed(5)
    kc = torch.randn(12, 16, 8, 128, generator=g).to(torch.bfloat16)
    vc = torch.randn(12, 16, 8, 128, generator=g).to(torch.bfloat16)
    src, dst, nv = [3, 7, 0], [9, 1, 5], [2, 16, 0]
    want_k, want_v = kc.clone(), vc.clone()
    for s, d, n in zip(src, dst, nv):
        want_k[d, :n] = kc[s, :n]
        want_v[d, :n] = vc[s, :n]
    dk, dv = kc.cuda(), vc.cuda()
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device="cuda")  # noqa: E731
    pa.pa_copy_blocks(dk, dv, i32(src), i32(dst), i32(nv))
    assert torch.equal(dk.cpu(), want_k) and torch.equal(dv.cpu(), want_v)


def _decode_direct(q, kc, vc, bt, ctx, max_ctx, scale, err=None):
    ws = pa.new_decode_workspace(q.shape[0], q.shape[1], kc.shape[2], q.shape[2], kc.shape[1], max_ctx)
    return pa.pa_decode(q, kc, vc, bt, ctx, max_ctx, scale, ws, error_count=err)


def test_long_single_sequence_fp32_many_partitions():
    """One fp32 sequence long enough to be split into many partitions: the
    cross-partition merge must keep fp32 accuracy."""
    rng = np.random.default_rng(11)
    L, B, Hq, Hkv, D = 9000, 16, 8, 2, 64
    nblk = oracle.num_blocks(L, B)
    P = nblk + 17
    table = rng.permutation(P)[:nblk].astype(np.int32)[None]
    kc = rng.standard_normal((P, B, Hkv, D), dtype=np.float32)
    vc = rng.standard_normal((P, B, Hkv, D), dtype=np.float32)
    q = rng.standard_normal((1, Hq, D), dtype=np.float32)
    want = oracle.decode(q, kc, vc, table, np.array([L], np.int32), 0.125)
    got = _decode_direct(*(torch.from_numpy(x).cuda() for x in (q, kc, vc, table, np.array([L], np.int32))), L, 0.125)
    assert _maxabs(got, want) <= 1e-5


@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-6), (torch.bfloat16, 1e-2)])
def test_split_count_does_not_change_the_result(dtype, tol):
    """The split-KV merge is exact up to rounding: one sequence decoded alone (its plan shrinks the partitions
    to cover the GPU: 64-token partitions, about 47 partials to merge) and as one member of a 64-sequence
    batch (768-token partitions, 4 partials) agree within `tol`."""
    rng = np.random.default_rng(12)
    N, L, B, Hq, Hkv, D = 64, 3000, 16, 8, 2, 128
    nblk = oracle.num_blocks(L, B)
    P = N * nblk + 9
    tables = rng.permutation(P)[:N * nblk].astype(np.int32).reshape(N, nblk)
    kc = torch.from_numpy(rng.standard_normal((P, B, Hkv, D), dtype=np.float32)).to(dtype).cuda()
    vc = torch.from_numpy(rng.standard_normal((P, B, Hkv, D), dtype=np.float32)).to(dtype).cuda()
    q = torch.from_numpy(rng.standard_normal((N, Hq, D), dtype=np.float32)).to(dtype).cuda()
    lens = torch.from_numpy(rng.integers(1, L + 1, size=N).astype(np.int32))
    lens[5] = L
    bt, ctx = torch.from_numpy(tables).cuda(), lens.cuda()
    part_one, splits_one = pa.pa_decode_plan(1, Hq, Hkv, D, B, L)
    part_all, splits_all = pa.pa_decode_plan(N, Hq, Hkv, D, B, L)
    # sequence 5 is not among the batch's last fifth: in the batch it has ceil(3000 / part_all) partitions
    assert splits_one > 40 and -(-L // part_all) <= 4
    alone = _decode_direct(q[5:6].contiguous(), kc, vc, bt[5:6].contiguous(), ctx[5:6].contiguous(), L, 0.09)
    batch = _decode_direct(q, kc, vc, bt, ctx, L, 0.09)
    torch.cuda.synchronize()
    assert float((alone[0].float() - batch[5].float()).abs().max()) <= tol


@pytest.mark.parametrize("N", [2, 4, 6])
def test_small_batches_shrink_partitions_in_multiples_of_64(N):
    """Small bf16 batches: the plan halves the partitions until the items cover the GPU twice (768 -> 384 ->
    192 -> 64 tokens, every length and its quarter-length tail a multiple of 64), and the decode still
    matches the oracle."""
    rng = np.random.default_rng(40 + N)
    Hq, Hkv, D, B = 32, 8, 128, 16
    lens = rng.integers(2500, 4097, size=N).astype(np.int32)
    part, splits = pa.pa_decode_plan(N, Hq, Hkv, D, B, int(lens.max()))
    assert part % 64 == 0 and part < 768 and splits >= -(-int(lens.max()) // part)
    nblk = [oracle.num_blocks(int(L), B) for L in lens]
    P = sum(nblk) + 11
    perm = rng.permutation(P).astype(np.int32)
    width = max(nblk)
    bt = np.full((N, width), -1, np.int32)
    o = 0
    for i, n in enumerate(nblk):
        bt[i, :n] = perm[o:o + n]
        o += n
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)  # noqa: E731
    q, kc, vc = (bf(rng.standard_normal(sh, dtype=np.float32)) for sh in ((N, Hq, D), (P, B, Hkv, D), (P, B, Hkv, D)))
    want = oracle.decode(storage_numpy(q), storage_numpy(kc), storage_numpy(vc), bt, lens, 1 / math.sqrt(D))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode_direct(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(),
                         int(lens.max()), 1 / math.sqrt(D), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _maxabs(got, want) <= TOL[torch.bfloat16]


def test_empty_and_single_token_contexts():
    rng = np.random.default_rng(3)
    P, B, Hq, Hkv, D = 8, 16, 8, 2, 128
    kc = rng.standard_normal((P, B, Hkv, D), dtype=np.float32)
    vc = rng.standard_normal((P, B, Hkv, D), dtype=np.float32)
    q = rng.standard_normal((3, Hq, D), dtype=np.float32)
    bt = np.array([[4, -1], [-1, -1], [2, 6]], np.int32)
    ctx = np.array([1, 0, 17], np.int32)
    for dt in (torch.float32, torch.bfloat16):
        t = lambda x: torch.from_numpy(x).to(dt).cuda()  # noqa: E731
        qd, kd, vd = t(q), t(kc), t(vc)
        # the oracle reads the same stored values (bf16 bit patterns for bf16)
        want = oracle.decode(storage_numpy(qd), storage_numpy(kd), storage_numpy(vd), bt, ctx, 0.1)
        got = _decode_direct(qd, kd, vd, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), 17, 0.1)
        assert torch.all(got[1] == 0)
        assert _maxabs(got, want) <= TOL[dt]
        # one token: the output is that token's V row exactly (bf16 V rows are representable in bf16)
        assert torch.equal(got[0].cpu(), vd[4, 0].cpu().repeat_interleave(4, 0))


def test_invalid_table_entries_are_skipped_and_counted():
    rng = np.random.default_rng(4)
    P, B, Hq, Hkv, D = 8, 16, 4, 4, 64
    kc = torch.from_numpy(rng.standard_normal((P, B, Hkv, D), dtype=np.float32)).cuda()
    q = torch.from_numpy(rng.standard_normal((2, Hq, D), dtype=np.float32)).cuda()
    bt = torch.tensor([[1, -1, 99], [2, 3, 4]], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([40, 200], dtype=torch.int32, device="cuda")  # seq 1 exceeds its table: clamped
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _decode_direct(q, kc, kc, bt, ctx, 48, 0.1, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) > 0
    assert torch.all(torch.isfinite(out))


def test_shared_prefix_branches_identical_after_device_cow():
    """Two branches share a 2050-token prefix whose last block is partial; the
    first branch's write copies it on the device (pa_copy_blocks).  With equal
    new tokens and equal queries both branches must give identical outputs."""
    B, Hq, Hkv, D = 16, 32, 8, 128
    alloc = BlockAllocator(200, B, seed=9)
    root = alloc.allocate(2050)
    b1, b2 = alloc.fork(root), alloc.fork(root)
    alloc.free(root)
    copies = alloc.append(b1, 1) + alloc.append(b2, 1)
    assert len(copies) == 1 and copies[0].num_valid == 2
    g = torch.Generator().manual_seed(2)
    kc = torch.randn(200, B, Hkv, D, generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn(200, B, Hkv, D, generator=g).to(torch.bfloat16).cuda()
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device="cuda")  # noqa: E731
    pa.pa_copy_blocks(kc, vc, i32([c.src for c in copies]), i32([c.dst for c in copies]),
                      i32([c.num_valid for c in copies]))
    bt = torch.from_numpy(alloc.block_table([b1, b2])).cuda()
    assert not torch.equal(bt[0], bt[1])  # the tails live in different physical blocks
    seq_idx, pos = i32([0, 1]), i32([2050, 2050])
    kn = torch.randn(1, Hkv, D, generator=g).to(torch.bfloat16).cuda().repeat(2, 1, 1)
    vn = torch.randn(1, Hkv, D, generator=g).to(torch.bfloat16).cuda().repeat(2, 1, 1)
    slots = pa.pa_slot_mapping(bt, seq_idx, pos, B, 200)
    pa.pa_write_kv(kn, vn, kc, vc, slots)
    q = torch.randn(1, Hq, D, generator=g).to(torch.bfloat16).cuda().repeat(2, 1, 1)
    out = _decode_direct(q, kc, vc, bt, i32([2051, 2051]), 2051, 1 / math.sqrt(D))
    assert torch.equal(out[0], out[1])


PREFILL_CASES = [
    # (Hq, Hkv, B, chunk_lens, offsets, dtype)
    (32, 8, 32, [512, 200], [0, 700], torch.bfloat16),
    (64, 8, 16, [129, 1, 33], [5, 0, 1000], torch.bfloat16),
    (8, 8, 64, [300], [64], torch.bfloat16),
    (16, 8, 128, [77, 256], [130, 0], torch.bfloat16),
    (32, 8, 8, [96], [1500], torch.bfloat16),
    (8, 4, 16, [70, 9], [3, 40], torch.float32),
]


DECODE_SHAPE_CASES = [
    # (Hq, Hkv, D, B, decode context lengths, dtype): tensor-core decode at head_dim 64 and 128, every block
    # size it takes and groups 1..8, stage and partition boundaries (63/64/65, 512/513, 1025, 4097), and the
    # CUDA-core path for group 16 and fp32
    (8, 8, 64, 16, [1, 63, 64, 65, 700, 1300], torch.bfloat16),
    (16, 8, 64, 8, [5, 512, 513, 2000], torch.bfloat16),
    (64, 8, 128, 64, [1, 100, 4097], torch.bfloat16),
    (32, 16, 128, 32, [3000, 17], torch.bfloat16),
    (16, 2, 128, 8, [1025, 64], torch.bfloat16),
    (128, 8, 128, 16, [300, 1], torch.bfloat16),
    (8, 2, 128, 16, [9000, 33], torch.float32),
    # block sizes only the CUDA-core kernel takes (1, 48, 128 on bf16 pools; 256 and 1024 on fp32 pools), with
    # contexts one short of, at and one past a block boundary
    (8, 2, 128, 1, [1, 300, 1100], torch.bfloat16),
    (32, 8, 128, 48, [47, 48, 49, 2000], torch.bfloat16),
    (16, 4, 64, 128, [127, 129, 1300], torch.bfloat16),
    (8, 8, 128, 256, [255, 257, 1024], torch.float32),
    (4, 2, 64, 1024, [1023, 1025, 3000], torch.float32),
]


@pytest.mark.parametrize("case", range(len(DECODE_SHAPE_CASES)))
def test_decode_shapes(case):
    Hq, Hkv, D, B, lens, dt = DECODE_SHAPE_CASES[case]
    w = W.prefill_batch(200 + case, Hq, Hkv, D, B, [], [], dtype=dt, decode_lens=lens)
    exp = expected_step(w)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    err = _maxabs(st.out_decode, exp.out_decode)
    assert err <= TOL[dt], f"decode max-abs error {err}"
    assert st.errors() == 0


@pytest.mark.parametrize("case", range(len(PREFILL_CASES)))
def test_prefill_shapes(case):
    Hq, Hkv, B, lens, offs, dt = PREFILL_CASES[case]
    w = W.prefill_batch(100 + case, Hq, Hkv, 128, B, lens, offs, dtype=dt, decode_lens=[1, 37])
    exp = expected_step(w)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    err = _maxabs(st.out_prefill, exp.out_prefill)
    assert err <= TOL[dt], f"prefill max-abs error {err}"
    assert _maxabs(st.out_decode, exp.out_decode) <= TOL[dt]
    assert st.errors() == 0


PREFILL_FALLBACK_CASES = [
    # (Hq, Hkv, D, B, chunk_lens, offsets, dtype): shapes the tensor-core prefill does not take (16 query heads
    # per kv head, head_dim 64), served by the CUDA-core prefill kernel
    (32, 2, 128, 16, [70, 1, 130], [3, 0, 300], torch.bfloat16),
    (16, 4, 64, 32, [200, 33], [0, 517], torch.bfloat16),
    (8, 8, 64, 16, [65, 9], [100, 0], torch.float32),
]


@pytest.mark.parametrize("case", range(len(PREFILL_FALLBACK_CASES)))
def test_prefill_fallback_shapes(case):
    Hq, Hkv, D, B, lens, offs, dt = PREFILL_FALLBACK_CASES[case]
    w = W.prefill_batch(140 + case, Hq, Hkv, D, B, lens, offs, dtype=dt, decode_lens=[2, 150])
    exp = expected_step(w)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    assert _maxabs(st.out_prefill, exp.out_prefill) <= TOL[dt]
    assert _maxabs(st.out_decode, exp.out_decode) <= TOL[dt]
    assert st.errors() == 0


PREFILL_RAGGED_CASES = [
    # (Hq, Hkv, B): many chunks of ragged lengths (one empty, single queries, a full 512) at scattered offsets,
    # so the persistent prefill grid walks several passes of items, most of them partial tiles
    (32, 8, 16),
    (64, 8, 64),
    (8, 8, 128),
]


@pytest.mark.parametrize("case", range(len(PREFILL_RAGGED_CASES)))
def test_prefill_many_ragged_chunks(case):
    Hq, Hkv, B = PREFILL_RAGGED_CASES[case]
    lens = [1, 0, 200, 33, 129, 7, 512, 64, 300, 5, 1, 96]
    offs = [0, 10, 700, 0, 2000, 64, 0, 3000, 1, 31, 4095, 128]
    w = W.prefill_batch(160 + case, Hq, Hkv, 128, B, lens, offs, dtype=torch.bfloat16, decode_lens=[3, 900])
    exp = expected_step(w)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    err = _maxabs(st.out_prefill, exp.out_prefill)
    assert err <= TOL[torch.bfloat16], f"prefill max-abs error {err}"
    assert _maxabs(st.out_decode, exp.out_decode) <= TOL[torch.bfloat16]
    assert st.errors() == 0


def test_graph_replay_matches_eager():
    """The captured step (CUDA graph of the four library calls) gives the same
    outputs as eager calls, replay after replay."""
    w, _ = _case("small", "mixed_bf16")
    st = DeviceStep(w)
    want = [t.clone() for t in st.run()]
    st.capture()
    for _ in range(3):
        got = st.replay()
        torch.cuda.synchronize()
        for x, y in zip(want, got):
            assert torch.equal(x, y)


def test_run_from_host_matches_device_step():
    """A step served from pinned host memory (one packed copy in, the step,
    one packed copy out) returns what the device step returns, eager or from
    the captured graph; new inputs written into the pinned buffer reach the
    kernels."""
    w, _ = _case("small", "mixed_bf16")
    st = DeviceStep(w)
    want = [t.clone() for t in st.run()]
    host_in, host_out = st.pinned_inputs(), st.pinned_outputs()
    st.step_from_host(host_in, host_out)
    st.capture_from_host(host_in, host_out)
    for graph in (False, True):
        host_out.zero_()
        st.run_from_host(host_in, host_out, graph=graph)
        torch.cuda.synchronize()
        for x, y in zip(want, st.output_views(host_out)):
            assert torch.equal(x.cpu(), y)
    st.input_views(host_in)["q_decode"].neg_()
    st.input_views(host_in)["q_prefill"].mul_(0.5)
    st.run_from_host(host_in, host_out, graph=True)
    torch.cuda.synchronize()
    fresh = [t.clone() for t in st.run()]  # eager, on the inputs the copy brought in
    assert not torch.equal(fresh[0], want[0])
    for x, y in zip(fresh, st.output_views(host_out)):
        assert torch.equal(x.cpu(), y)


def test_decode_plan_matches_workspace_and_launches():
    """The plan reported through the ABI is the one pa_decode sizes its
    workspace for: 768-token partitions on the bf16 decode workload (64
    sequences, 8 kv heads, contexts up to 4096), with room for the
    quarter-length partitions of the batch's last sequences (22 slots); a
    context that fits one partition has one, and two quarter-length ones at
    most."""
    part, splits = pa.pa_decode_plan(64, 32, 8, 128, 16, 4096)
    assert (part, splits) == (768, 22)
    need = pa.pa_decode_workspace_size(64, 32, 8, 128, 16, 4096)
    assert need >= 64 * 8 * splits * 4 * 128 * 4
    part1, splits1 = pa.pa_decode_plan(512, 32, 8, 128, 16, 300)
    assert part1 >= 300 and splits1 == 2


@pytest.mark.parametrize("prefix_len,B", [(100, 16), (2048, 16), (160, 32)])
def test_cascade_decode_matches_oracle_and_plain_decode(prefix_len, B):
    """Cascade decode (each group's shared prefix read once, on the tensor
    cores, merged with every member's private tail) against the oracle and
    against plain paged decode of the same batch.  A 100-token prefix leaves
    96 tokens in shared full blocks (not a multiple of 64: the tail pass masks
    tokens 64..95 of its first stage) and the copied partial block in the tails."""
    w = W.shared_prefix_bf16(3, num_prompts=3, branches=5, prefix_len=prefix_len, max_tail=70, B=B,
                             name="cascade_case")
    assert int(w.prefix_lens.max()) > 0
    exp = expected_step(w)
    cas = DeviceStep(w)
    assert cas.use_cascade
    cas.slot_mapping()
    cas.write_kv()
    got = cas.decode().clone()
    plain = DeviceStep(w, cascade=False)
    plain.run()
    torch.cuda.synchronize()
    assert cas.errors() == 0 and plain.errors() == 0
    assert _maxabs(got, exp.out_decode) <= TOL[w.dtype]
    assert (got.float() - plain.out_decode.float()).abs().max().item() <= TOL[w.dtype]
    # repeat: bitwise identical
    again = cas.decode()
    torch.cuda.synchronize()
    assert torch.equal(again, got)


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 8), (16, 4)])
def test_cascade_decode_every_head_group(Hq, Hkv):
    """Cascade decode with 8, 1 and 4 query heads per kv head: a group's tile holds 32 / G members' rows, so
    with G = 8 the five branches of a prompt split into groups of four and one, and with G = 1 they share one
    five-row tile.  Against the oracle and against plain decode of the same batch."""
    w = W.shared_prefix_bf16(11, num_prompts=3, branches=5, prefix_len=100, max_tail=60, B=16, name="cascade_heads",
                             num_q_heads=Hq, num_kv_heads=Hkv)
    exp = expected_step(w)
    cas = DeviceStep(w)
    assert cas.use_cascade
    cas.slot_mapping()
    cas.write_kv()
    got = cas.decode().clone()
    plain = DeviceStep(w, cascade=False)
    plain.run()
    torch.cuda.synchronize()
    assert cas.errors() == 0 and plain.errors() == 0
    assert _maxabs(got, exp.out_decode) <= TOL[w.dtype]
    assert (got.float() - plain.out_decode.float()).abs().max().item() <= TOL[w.dtype]


@pytest.mark.parametrize("name", ["tiny_fp32", "mixed_bf16", "shared_prefix_bf16"])
def test_fused_slot_mapping_and_write_matches_oracle(name):
    """pa_write_kv_paged (slot mapping and scatter in one launch) writes exactly
    the pools and slots the oracle's two steps give."""
    w, exp = _case("small", name)
    st = DeviceStep(w)
    st.write_kv_paged()
    torch.cuda.synchronize()
    assert torch.equal(st.slots.cpu(), torch.from_numpy(exp.slots))
    assert np.array_equal(storage_numpy(st.k_cache.cpu()), exp.k_cache)
    assert np.array_equal(storage_numpy(st.v_cache.cpu()), exp.v_cache)
    assert st.errors() == 0


def test_fused_write_counts_invalid_entries_like_slot_mapping():
    bt = torch.tensor([[3, -1], [0, 1]], dtype=torch.int32, device="cuda")
    seq = torch.tensor([0, 0, 1, 1, 0, 2, -1, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([5, -1, 9, 20, 17, 0, 0, 40], dtype=torch.int32, device="cuda")
    kc = torch.zeros(4, 16, 2, 8, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.arange(1, 8 * 16 + 1, dtype=torch.float32, device="cuda").view(8, 2, 8).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.empty(8, dtype=torch.int64, device="cuda")
    pa.pa_write_kv_paged(kn, -kn, kc, vc, bt, seq, pos, slot_mapping=slots, error_count=err)
    want, nerr = oracle.slot_mapping(bt.cpu().numpy(), seq.cpu().numpy(), pos.cpu().numpy(), 16, 4)
    assert slots.cpu().tolist() == want.tolist() and int(err.item()) == nerr
    flat_k, flat_v = kc.view(64, 16), vc.view(64, 16)
    for t, sl in enumerate(want.tolist()):
        if sl >= 0:
            assert torch.equal(flat_k[sl], kn[t].view(16)) and torch.equal(flat_v[sl], -kn[t].view(16))
    assert torch.count_nonzero(flat_k).item() == 16 * sum(1 for x in want.tolist() if x >= 0)


def test_stage_copy_moves_bytes_between_pinned_host_and_device():
    g = torch.Generator().manual_seed(9)
    host = torch.randint(0, 256, (1 << 20,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    pa.pa_stage_copy(dev, host)
    back = torch.zeros(1 << 20, dtype=torch.uint8).pin_memory()
    pa.pa_stage_copy(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host) and torch.equal(back, host)
    with pytest.raises(ValueError):  # pageable host memory is refused before anything is launched
        pa.pa_stage_copy(dev, torch.zeros(1 << 20, dtype=torch.uint8))


def test_cascade_groups_wider_than_a_tile_use_the_prefill_prefix_pass():
    """A group of 12 sequences x 4 heads (48 query rows) is more than the
    decode kernel's 32-row tile: pa_decode_cascade reads its prefix with the
    tensor-core prefill kernel's prefix pass instead; same results."""
    w = W.shared_prefix_bf16(7, num_prompts=2, branches=12, prefix_len=160, max_tail=50, B=16, name="wide_groups")
    exp = expected_step(w)
    st = DeviceStep(w, cascade=False)
    st.write_kv_paged()
    nd = w.num_decode
    offs = torch.tensor([0, 12, 24], dtype=torch.int32, device="cuda")
    pre = torch.full((nd,), 160, dtype=torch.int32, device="cuda")
    ws = pa.new_cascade_workspace(nd, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, st.max_context_len)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pa.pa_decode_cascade(st.q_decode, st.k_cache, st.v_cache, st.block_tables[:nd], st.context_lens[:nd],
                               st.max_context_len, offs, 12, pre, w.scale, ws, error_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _maxabs(got, exp.out_decode) <= TOL[w.dtype]


def test_map_to_kernel_blocks_matches_oracle_and_decode_through_it():
    """Manager blocks of 64 tokens (4 kernel blocks of 16): the device remap equals the oracle's, and
    decode through the remapped table on the same pool gives the oracle's decode through the manager
    table (the pool [P][64][Hkv][D] read as [4P][16][Hkv][D])."""
    rng = np.random.default_rng(31)
    ratio, Bk, Hq, Hkv, D = 4, 16, 32, 8, 128
    Bm = ratio * Bk
    lens = np.array([1, 64, 65, 700, 2000, 333], np.int32)
    nb = -(-lens // Bm)
    P = int(nb.sum()) + 3
    perm = rng.permutation(P).astype(np.int32)
    mgr = np.full((len(lens), int(nb.max())), -1, np.int32)
    at = 0
    for s, n in enumerate(nb):
        mgr[s, :n] = perm[at:at + n]
        at += n
    kc = rng.standard_normal((P, Bm, Hkv, D), dtype=np.float32)
    vc = rng.standard_normal((P, Bm, Hkv, D), dtype=np.float32)
    q = rng.standard_normal((len(lens), Hq, D), dtype=np.float32)
    want_tables = oracle.map_to_kernel_blocks(mgr, ratio)
    got_tables = pa.pa_map_to_kernel_blocks(torch.from_numpy(mgr).cuda(), ratio)
    assert np.array_equal(got_tables.cpu().numpy(), want_tables)
    want = oracle.decode(q, kc, vc, mgr, lens, 1.0 / math.sqrt(D))  # manager view, block size 64
    bf = lambda x: torch.from_numpy(x).to(torch.bfloat16).cuda()  # noqa: E731
    kk = bf(kc).view(P * ratio, Bk, Hkv, D)
    vv = bf(vc).view(P * ratio, Bk, Hkv, D)
    want_bf = oracle.decode(bf(q).float().cpu().numpy(), bf(kc).float().cpu().numpy(),
                            bf(vc).float().cpu().numpy(), mgr, lens, 1.0 / math.sqrt(D))
    got = _decode_direct(bf(q), kk, vv, got_tables, torch.from_numpy(lens).cuda(), int(lens.max()),
                         1.0 / math.sqrt(D))
    assert _maxabs(got, want_bf) <= TOL[torch.bfloat16]
    assert np.abs(want_bf - want).max() < 0.1  # bf16 inputs vs fp32 inputs: same attention


def test_multi_layer_pools_share_one_slot_mapping():
    """A 3-layer pool [layers][P][B][Hkv][D] ("KV cache 显存管理…": the cache is per layer, the block table
    is not): one slot mapping per step, then per layer the write and the decode on that layer's slice,
    each equal to the oracle's on that layer."""
    w, _ = _case("small", "decode_bf16")
    layers = 3
    rng = np.random.default_rng(41)
    P, B, Hkv, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    nd, T = w.num_decode, int(w.seq_idx.numel())
    mk = lambda *shape: torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)  # noqa
    kpool, vpool = mk(layers, P, B, Hkv, D), mk(layers, P, B, Hkv, D)
    knew, vnew, q = mk(layers, T, Hkv, D), mk(layers, T, Hkv, D), mk(layers, nd, w.num_q_heads, D)
    dk, dv = kpool.cuda(), vpool.cuda()
    bt, ctx = w.block_tables.cuda(), w.context_lens.cuda()
    slots = pa.pa_slot_mapping(bt, w.seq_idx.cuda(), w.pos.cuda(), B, P)
    for layer in range(layers):
        pa.pa_write_kv(knew[layer].cuda(), vnew[layer].cuda(), dk[layer], dv[layer], slots)
        got = _decode_direct(q[layer].cuda(), dk[layer], dv[layer], bt[:nd], ctx[:nd], w.max_decode_context,
                             w.scale)
        kc, vc = storage_numpy(kpool[layer]).copy(), storage_numpy(vpool[layer]).copy()
        sl, _ = oracle.slot_mapping(w.block_tables.numpy(), w.seq_idx.numpy(), w.pos.numpy(), B, P)
        oracle.write_kv(storage_numpy(knew[layer]), storage_numpy(vnew[layer]), kc, vc, sl)
        assert np.array_equal(storage_numpy(dk[layer].cpu()), kc)
        want = oracle.decode(storage_numpy(q[layer]), kc, vc, w.block_tables.numpy()[:nd],
                             w.context_lens.numpy()[:nd], w.scale)
        assert _maxabs(got, want) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("name", ["decode_bf16", "mixed_bf16", "longctx_bf16"])
def test_decode_write_equals_separate_write_then_decode(name):
    """pa_decode_write (the decode kernel writes each sequence's newest token into the pool and attends with
    it) leaves the same pools and slots as the separate write and gives the same outputs, bit for bit."""
    w, exp = _case("small", name)
    fused = DeviceStep(w)
    assert fused.fused_decode_write
    plain = DeviceStep(w, fused_decode_write=False)
    fused.run()
    plain.run()
    torch.cuda.synchronize()
    assert fused.errors() == 0 and plain.errors() == 0
    assert torch.equal(fused.slots.cpu(), torch.from_numpy(exp.slots))
    assert np.array_equal(storage_numpy(fused.k_cache.cpu()), exp.k_cache)
    assert np.array_equal(storage_numpy(fused.v_cache.cpu()), exp.v_cache)
    assert torch.equal(fused.out_decode, plain.out_decode)
    assert torch.equal(fused.out_prefill, plain.out_prefill)
    assert _maxabs(fused.out_decode, exp.out_decode) <= TOL[w.dtype]


# ---- e4m3 pools ------------------------------------------------------------

@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 0.37), (1.0 / 64, 3.0)])
def test_fp8_write_of_every_bf16_value_matches_oracle(k_scale, v_scale):
    """The quantising write, bit-exact against the oracle's nearest-code search, for every bf16 bit pattern but
    the NaNs (64 tokens x 8 heads x 128 = 65536 elements; infinities saturate), at power-of-two scales and at
    scales whose reciprocal and product round; whole pools compared, untouched slots included."""
    T, H, D, B, P = 64, 8, 128, 16, 9
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bits[((bits & 0x7F80) == 0x7F80) & ((bits & 0x7F) != 0)] = 0
    rng = np.random.default_rng(11)
    k_bits = bits.reshape(T, H, D)
    v_bits = rng.permutation(bits).reshape(T, H, D)
    bt = np.array([[7, 2, 5, 0]], dtype=np.int32)
    seq_idx = np.zeros(T, dtype=np.int32)
    pos = np.arange(T, dtype=np.int32)
    kc0 = rng.integers(0, 256, size=(P, B, H, D), dtype=np.uint8)
    vc0 = rng.integers(0, 256, size=(P, B, H, D), dtype=np.uint8)
    slots, nerr = oracle.slot_mapping(bt, seq_idx, pos, B, P)
    assert nerr == 0
    k_exp, v_exp = kc0.copy(), vc0.copy()
    assert oracle.write_kv_fp8(k_bits, v_bits, k_exp, v_exp, slots, k_scale, v_scale) == 0

    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    bf = lambda b: dev(b.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    kc, vc = dev(kc0), dev(vc0)
    slot_out = torch.empty(T, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv_paged_fp8(bf(k_bits), bf(v_bits), kc, vc, dev(bt), dev(seq_idx), dev(pos), k_scale, v_scale,
                             slot_mapping=slot_out, error_count=err)
    torch.cuda.synchronize()
    assert torch.equal(slot_out.cpu(), torch.from_numpy(slots))
    assert np.array_equal(kc.cpu().numpy(), k_exp), "K codes differ"
    assert np.array_equal(vc.cpu().numpy(), v_exp), "V codes differ"
    assert int(err.item()) == 0


@pytest.mark.parametrize("kind", ["small", "full"])
def test_decode_write_fp8_equals_separate_write_then_decode(kind):
    """pa_decode_write_fp8 (the e4m3 decode kernel quantises each sequence's newest token, stores the codes in the
    pools and attends with them) leaves the same pools and slots as the separate quantising write and gives the
    same outputs, bit for bit, at the step's full size and reduced."""
    w, exp = _case(kind, "decode_fp8")
    fused = DeviceStep(w)
    assert fused.fused_decode_write
    plain = DeviceStep(w, fused_decode_write=False)
    fused.run()
    plain.run()
    torch.cuda.synchronize()
    assert fused.errors() == 0 and plain.errors() == 0
    assert torch.equal(fused.slots.cpu(), torch.from_numpy(exp.slots))
    assert torch.equal(fused.k_cache, plain.k_cache) and torch.equal(fused.v_cache, plain.v_cache)
    assert np.array_equal(fused.k_cache.cpu().numpy(), exp.k_cache)
    assert np.array_equal(fused.v_cache.cpu().numpy(), exp.v_cache)
    assert torch.equal(fused.out_decode, plain.out_decode)
    assert _maxabs(fused.out_decode, exp.out_decode) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 0.37), (1.0 / 64, 3.0), (0.7, 0.9), (0.6, 1.0)])
def test_fused_fp8_write_of_every_bf16_value_matches_oracle(k_scale, v_scale):
    """The quantising write inside the e4m3 decode kernel, bit-exact against the oracle for every bf16 bit pattern
    but the NaNs: 64 sequences x 8 kv heads x 128 columns of newest-token K (and a permutation for V) = 65536
    elements, at power-of-two scales and at scales whose reciprocal and product round.  Whole pools compared
    (untouched slots included); the outputs bit-identical to the separate quantising write followed by
    pa_decode_fp8 (the codes span the whole e4m3 range here, so outputs reach magnitudes where the absolute bf16
    tolerance of the workloads does not apply)."""
    N, Hq, H, D, B = 64, 32, 8, 128, 16
    rng = np.random.default_rng(17)
    lens = (1 + 5 * np.arange(N)).astype(np.int32)  # the newest token lands at every offset of a block
    nblk = [oracle.num_blocks(int(L), B) for L in lens]
    P = sum(nblk) + 7
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((N, max(nblk)), -1, np.int32)
    o = 0
    for s_, nb in enumerate(nblk):
        bt[s_, :nb] = perm[o:o + nb]
        o += nb
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bits[((bits & 0x7F80) == 0x7F80) & ((bits & 0x7F) != 0)] = 0
    k_bits = bits.reshape(N, H, D)
    v_bits = rng.permutation(bits).reshape(N, H, D)
    kc0 = (rng.integers(0x30, 0x60, size=(P, B, H, D), dtype=np.uint8) | (rng.integers(0, 2, size=(P, B, H, D), dtype=np.uint8) << 7))
    vc0 = (rng.integers(0x30, 0x60, size=(P, B, H, D), dtype=np.uint8) | (rng.integers(0, 2, size=(P, B, H, D), dtype=np.uint8) << 7))
    slots, nerr = oracle.slot_mapping(bt, np.arange(N, dtype=np.int32), lens - 1, B, P)
    assert nerr == 0
    k_exp, v_exp = kc0.copy(), vc0.copy()
    assert oracle.write_kv_fp8(k_bits, v_bits, k_exp, v_exp, slots, k_scale, v_scale) == 0
    q = torch.from_numpy(rng.standard_normal((N, Hq, D), dtype=np.float32)).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    bf = lambda b: dev(b.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    kc, vc = dev(kc0), dev(vc0)
    slot_out = torch.full((N,), -7, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pa.new_decode_workspace(N, Hq, H, D, B, int(lens.max()))
    out = pa.pa_decode_write_fp8(q.cuda(), kc, vc, dev(bt), dev(lens), int(lens.max()), scale, k_scale, v_scale,
                                 bf(k_bits), bf(v_bits), ws, new_slots=slot_out, error_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(slot_out.cpu(), torch.from_numpy(slots))
    assert np.array_equal(kc.cpu().numpy(), k_exp), "K codes differ"
    assert np.array_equal(vc.cpu().numpy(), v_exp), "V codes differ"
    kc2, vc2 = dev(kc0), dev(vc0)
    pa.pa_write_kv_paged_fp8(bf(k_bits), bf(v_bits), kc2, vc2, dev(bt), dev(np.arange(N, dtype=np.int32)),
                             dev(lens - 1), k_scale, v_scale, error_count=err)
    ws2 = pa.new_decode_workspace(N, Hq, H, D, B, int(lens.max()))
    out2 = pa.pa_decode_fp8(q.cuda(), kc2, vc2, dev(bt), dev(lens), int(lens.max()), scale, k_scale, v_scale, ws2,
                            error_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)
    assert torch.equal(out, out2)


FP8_DECODE_CASES = [
    # (Hq, Hkv, B, decode context lengths, code range): every block size, groups 1..8, partition boundaries,
    # and codes over the whole finite range (subnormals up to 448) through the in-register conversion; even
    # kv-head counts run items of two kv heads
    (8, 8, 8, [1, 63, 64, 65, 700], (0x30, 0x60)),
    (16, 8, 16, [5, 512, 513, 2000], (0x30, 0x60)),
    (32, 8, 32, [3000, 17, 129], (0x30, 0x60)),
    (64, 8, 64, [1, 100, 4097], (0x30, 0x60)),
    (32, 8, 16, [900, 64, 1], (0x00, 0x7F)),
    (16, 2, 8, [1025, 64], (0x00, 0x7F)),
    (12, 3, 16, [700, 33, 1, 1200], (0x30, 0x60)),  # odd kv-head count: one kv head per item
]


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (32, 2, 128)])
def test_fp8_decode_refuses_shapes_it_does_not_build(Hq, Hkv, D):
    """Head size 64 and 16 query heads per kv head have no e4m3 kernel: the call returns PA_ERR_UNSUPPORTED (no
    launch, no silent fallback) although the same shapes over bf16 pools are served."""
    N, B, P = 2, 16, 8
    q = torch.zeros(N, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(P, B, Hkv, D, dtype=torch.uint8, device="cuda")
    bt = torch.arange(N * 2, dtype=torch.int32, device="cuda").view(N, 2)
    ctx = torch.tensor([5, 20], dtype=torch.int32, device="cuda")
    ws = pa.new_decode_workspace(N, Hq, Hkv, D, B, 20)
    with pytest.raises(pa.PaError) as ei:
        pa.pa_decode_fp8(q, kc, kc.clone(), bt, ctx, 20, 0.1, 1.0, 1.0, ws)
    assert ei.value.status == pa.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", range(len(FP8_DECODE_CASES)))
def test_fp8_decode_shapes(case):
    Hq, Hkv, B, lens, (lo, hi) = FP8_DECODE_CASES[case]
    w = W.prefill_batch(300 + case, Hq, Hkv, 128, B, [], [], dtype=torch.bfloat16, decode_lens=lens)
    ks, vs = (1.0 / 64, 1.0 / 64) if hi <= 0x60 else (1.0 / 256, 1.0 / 128)
    W.as_fp8(w, 300 + case, ks, vs, lo, hi)
    exp = expected_step(w)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    assert np.array_equal(storage_numpy(st.k_cache.cpu()), exp.k_cache)
    assert np.array_equal(storage_numpy(st.v_cache.cpu()), exp.v_cache)
    err = _maxabs(st.out_decode, exp.out_decode)
    assert err <= TOL[torch.bfloat16], f"fp8 decode max-abs error {err}"
    assert st.errors() == 0


def test_bounded_wait_gives_up_counts_an_error_and_leaves_the_context_usable():
    """The wait every kernel uses on its mbarriers is bounded: on a barrier nothing arrives on, it gives up
    after its poll limit, reports false and counts an error, and the kernel returns normally; with the arrival
    it succeeds.  The context stays usable: a decode right after matches the oracle."""
    assert pa.pa_check_bounded_wait(256, arrive=False) == (0, 1)
    assert pa.pa_check_bounded_wait(256, arrive=True) == (1, 0)
    assert pa.pa_check_bounded_wait(1, arrive=False) == (0, 1)
    w = W.tiny_fp32(0)
    exp = expected_step(w)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    assert _maxabs(st.out_decode, exp.out_decode) <= 1e-5
    assert st.errors() == 0


def test_cascade_counts_a_member_whose_table_breaks_the_group():
    """A group's prefix is read through its first member's table, so every member must map the same physical
    blocks over the prefix ("什么是 PagedAttention？", 共享但不污染状态).  A caller's group in which one member
    maps a different (valid) block inside the prefix is counted in error_count; the other sequences' outputs
    still match the oracle."""
    w = W.shared_prefix_bf16(3, num_prompts=3, branches=5, prefix_len=100, max_tail=70, B=16, name="cascade_bad")
    cas = DeviceStep(w)
    assert cas.use_cascade
    cas.slot_mapping()
    cas.write_kv()
    torch.cuda.synchronize()
    goff = w.group_offsets.tolist()
    s = goff[0] + 1  # the group's second member
    assert goff[1] - goff[0] >= 2 and int(w.prefix_lens[s]) >= 32
    bt = w.block_tables.clone()
    other = int(bt[goff[1], 0])  # a valid block of another prompt, not in this group's prefix
    assert other not in bt[goff[0], :4].tolist()
    bt[s, 1] = other
    cas.block_tables.copy_(bt.to(cas.block_tables.device))
    got = cas.decode().clone()
    torch.cuda.synchronize()
    assert cas.errors() >= 1
    nd = w.num_decode
    want = oracle.decode(storage_numpy(w.q_decode), storage_numpy(cas.k_cache.cpu()), storage_numpy(cas.v_cache.cpu()),
                         bt.numpy()[:nd], w.context_lens.numpy()[:nd], w.scale)
    keep = [i for i in range(nd) if i != s]
    assert _maxabs(got[keep], want[keep]) <= TOL[w.dtype]
    # the consistent batch counts nothing
    cas.block_tables.copy_(w.block_tables.to(cas.block_tables.device))
    cas.error_count.zero_()
    cas.decode()
    torch.cuda.synchronize()
    assert cas.errors() == 0
