"""Pins for the CPU oracle: what the pages print, closed forms, invariants and
brute force.  None of these re-type the oracle's own code path; each is built so
that a plausible slip (wrong index, dropped scale, transposed K/V, wrong KV-head
mapping, off-by-one context, missing causal limit) fails at least one test.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def _bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (test helper, storage form)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _place(contig, table, num_blocks, block_size):
    """Put a contiguous [L, Hkv, D] array into a fresh pool by the block table's
    meaning: logical block i holds tokens [iB, (i+1)B) and lives in physical
    block table[i].  Written with numpy block views, not with slot arithmetic."""
    L, H, D = contig.shape
    pool = np.full((num_blocks, block_size, H, D), np.nan, dtype=contig.dtype) if contig.dtype == np.float32 \
        else np.zeros((num_blocks, block_size, H, D), dtype=contig.dtype)
    for i, pb in enumerate(table):
        chunk = contig[i * block_size:(i + 1) * block_size]
        pool[pb, : chunk.shape[0]] = chunk
    return pool


# ------------------------------------------------------------------ golden
def test_worked_example_block_count_and_ranges(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example_b16.json")))
    B, L = g["block_size"], g["seq_len"]
    assert oracle.num_blocks(L, B) == g["num_blocks"]
    assert oracle.num_blocks(g["len17"]["seq_len"], B) == g["len17"]["num_blocks"]
    assert g["len17"]["seq_len"] - (g["len17"]["num_blocks"] - 1) * B == g["len17"]["tokens_in_last_block"]
    # every token of the 40-token sequence resolves to the printed block and its offset in it
    table = np.array([g["block_table"]], dtype=np.int32)
    pos = np.arange(L, dtype=np.int32)
    slots, err = oracle.slot_mapping(table, np.zeros(L, np.int32), pos, B, 16)
    assert err == 0
    for (lo, hi), pb in zip(g["valid_token_ranges"], g["block_table"]):
        for tok in range(lo, hi + 1):
            assert slots[tok] // B == pb and slots[tok] % B == tok - lo
    # the third block's capacity range 32..47 all lands in physical block 15
    cap_lo, cap_hi = g["capacity_token_ranges"][2]
    s, err = oracle.slot_mapping(table, np.zeros(cap_hi - cap_lo + 1, np.int32),
                                 np.arange(cap_lo, cap_hi + 1, dtype=np.int32), B, 16)
    assert err == 0 and np.all(s // B == 15) and list(s % B) == list(range(B))
    # token 33 -> logical block 2, offset 1 -> physical block 15
    s33, _ = oracle.slot_mapping(table, [0], [33], B, 16)
    assert (s33[0] // B, s33[0] % B) == (15, 1)


def test_tail_waste_bound(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example_b16.json")))
    B = g["block_size"]
    wastes = [oracle.num_blocks(L, B) * B - L for L in range(1, 5 * B + 3)]
    assert max(wastes) == g["max_tail_waste"] and min(wastes) == 0
    ex = g["kv_tokens_example"]
    assert ex["prompt"] + ex["generated"] == ex["total"]
    assert oracle.num_blocks(ex["total"], B) * B - ex["total"] <= g["max_tail_waste"]
    r = g["reservation_example"]
    assert r["reserved"] - r["used"] == r["wasted"]
    assert oracle.num_blocks(r["used"], B) * B - r["used"] < r["wasted"]


# ------------------------------------------------------- slot mapping / write
@pytest.mark.parametrize("B", [1, 2, 4, 16])
def test_slot_write_brute_force(B):
    """Every placement of up to 3 logical blocks in a 4-block pool, every length:
    writing a labelled contiguous sequence through the oracle's slot mapping and
    KV write must give the block-view placement."""
    P, H, D = 4, 2, 3
    for nblk in range(0, 4):
        for table in itertools.permutations(range(P), nblk):
            for L in range(max(0, (nblk - 1) * B + 1), nblk * B + 1):
                contig = (np.arange(L * H * D, dtype=np.float32) + 1).reshape(L, H, D)
                bt = np.array([list(table) + [-1] * (3 - nblk)], dtype=np.int32)
                slots, err = oracle.slot_mapping(bt, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), B, P)
                assert err == 0
                kc = np.full((P, B, H, D), np.nan, np.float32)
                vc = np.full((P, B, H, D), np.nan, np.float32)
                assert oracle.write_kv(contig, -contig, kc, vc, slots) == 0
                want = _place(contig, table, P, B)
                np.testing.assert_array_equal(kc, want)
                np.testing.assert_array_equal(vc, np.where(np.isnan(want), np.nan, -want))
                assert len(set(slots.tolist())) == L  # distinct slots for distinct tokens


def test_slot_mapping_padding_and_errors():
    bt = np.array([[3, -1], [0, 1]], dtype=np.int32)
    seq = np.array([0, 0, 1, 1, 0, 2, -1, 1], np.int32)
    pos = np.array([5, -1, 9, 20, 17, 0, 0, 40], np.int32)
    slots, err = oracle.slot_mapping(bt, seq, pos, 16, 4)
    # 5 -> block 3 off 5; pad; 9 -> block 0 off 9; 20 -> block 1 off 4;
    # 17 -> table entry -1 (error); seq 2 and -1 out of range (errors); 40 -> logical 2 >= width (error)
    assert slots.tolist() == [53, -1, 9, 20, -1, -1, -1, -1]
    assert err == 4


def test_write_kv_skips_negative_and_rejects_out_of_pool():
    kc = np.zeros((2, 4, 1, 2), np.float32)
    vc = np.zeros_like(kc)
    kn = np.ones((3, 1, 2), np.float32)
    err = oracle.write_kv(kn, 2 * kn, kc, vc, np.array([-1, 5, 8], np.int64))
    assert err == 1
    assert kc.reshape(8, 2)[5].tolist() == [1, 1] and vc.reshape(8, 2)[5].tolist() == [2, 2]
    assert np.count_nonzero(kc) == 2


# ------------------------------------------------------------- attention
def _decode_single(q, kc_contig, vc_contig, B, P, scale, seed=0, dtype=np.float32):
    """One sequence, one head group: scatter contiguous K/V to a random placement and decode."""
    L = kc_contig.shape[0]
    nblk = oracle.num_blocks(L, B)
    rng = np.random.default_rng(seed)
    table = rng.permutation(P)[:nblk]
    kp = _place(kc_contig, table, P, B)
    vp = _place(vc_contig, table, P, B)
    if dtype == np.float32:
        kp = np.nan_to_num(kp, nan=1e30)  # unused slots hold huge values a correct oracle never reads
        vp = np.nan_to_num(vp, nan=1e30)
    bt = np.array([list(table) + [-1]], dtype=np.int32)
    return oracle.decode(q[None], kp, vp, bt, np.array([L], np.int32), scale)[0]


def test_single_token_returns_its_value():
    D = 8
    q = RNG.standard_normal((1, D)).astype(np.float32)
    k = RNG.standard_normal((1, 1, D)).astype(np.float32)
    v = RNG.standard_normal((1, 1, D)).astype(np.float32)
    o = _decode_single(q, k, v, 16, 4, 0.3)
    np.testing.assert_array_equal(o[0], v[0, 0].astype(np.float64))


def test_two_token_closed_form():
    # x0 = 0.5 * (1*2 + 0*0) = 1, x1 = 0: weights e/(1+e) and 1/(1+e) (the logistic function)
    q = np.array([[1.0, 0.0]], np.float32)
    k = np.array([[[2.0, 0.0]], [[0.0, 0.0]]], np.float32)
    v = np.array([[[1.0, 0.0]], [[0.0, 1.0]]], np.float32)
    o = _decode_single(q, k, v, 1, 5, 0.5)[0]
    w0 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(o, [w0, 1.0 - w0], rtol=0, atol=1e-15)
    # swapping the roles of K and V must change the answer (guards a transposed operand)
    o_swapped = _decode_single(q, v, k, 1, 5, 0.5)[0]
    assert not np.allclose(o_swapped, o)


def test_equal_keys_and_zero_scale_give_mean():
    L, D = 37, 16
    q = RNG.standard_normal((1, D)).astype(np.float32)
    v = RNG.standard_normal((L, 1, D)).astype(np.float32)
    k_same = np.repeat(RNG.standard_normal((1, 1, D)).astype(np.float32), L, axis=0)
    mean = v[:, 0].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(_decode_single(q, k_same, v, 16, 8, 0.7)[0], mean, atol=1e-12)
    k = RNG.standard_normal((L, 1, D)).astype(np.float32)
    np.testing.assert_allclose(_decode_single(q, k, v, 4, 12, 0.0)[0], mean, atol=1e-12)


def test_dominant_key_selects_its_value():
    L, D = 20, 8
    k = RNG.standard_normal((L, 1, D)).astype(np.float32)
    v = RNG.standard_normal((L, 1, D)).astype(np.float32)
    q = k[13].copy() * 4
    o = _decode_single(q, k, v, 4, 8, 100.0)[0]
    np.testing.assert_allclose(o, v[13, 0], atol=1e-9)


def test_placement_order_shift_and_linearity_invariants():
    L, D = 45, 16
    q = RNG.standard_normal((1, D)).astype(np.float32)
    k = RNG.standard_normal((L, 1, D)).astype(np.float32)
    v = RNG.standard_normal((L, 1, D)).astype(np.float32)
    base = _decode_single(q, k, v, 16, 8, 0.25, seed=1)
    # placement: different block size and different random tables give the same answer
    for B, P, seed in [(1, 64, 2), (4, 20, 3), (16, 5, 4)]:
        np.testing.assert_allclose(_decode_single(q, k, v, B, P, 0.25, seed=seed), base, rtol=0, atol=1e-13)
    # token order does not matter for decode (no positional term)
    perm = RNG.permutation(L)
    np.testing.assert_allclose(_decode_single(q, k[perm], v[perm], 16, 8, 0.25), base, atol=1e-13)
    # adding one vector to every key shifts all scores equally
    u = RNG.standard_normal((1, 1, D)).astype(np.float32)
    shifted = (k.astype(np.float64) + u).astype(np.float32)
    ref = _decode_single(q, shifted, v, 16, 8, 0.25)
    # compare against the unshifted result computed on keys with the same fp32 rounding error budget
    np.testing.assert_allclose(ref, base, atol=1e-5)
    # linear in V
    v2 = RNG.standard_normal((L, 1, D)).astype(np.float32)
    o2 = _decode_single(q, k, v2, 16, 8, 0.25)
    o12 = _decode_single(q, k, (v.astype(np.float64) + v2).astype(np.float32), 16, 8, 0.25)
    np.testing.assert_allclose(o12, base + o2, atol=1e-6)


def test_independent_contiguous_attention():
    """Paged == contiguous: a second, numpy-only fp64 computation on the contiguous
    tensor (no block table involved) agrees with the oracle on a random placement."""
    L, D = 100, 32
    q = RNG.standard_normal((1, D)).astype(np.float32)
    k = RNG.standard_normal((L, 1, D)).astype(np.float32)
    v = RNG.standard_normal((L, 1, D)).astype(np.float32)
    s = 0.3 * (k[:, 0].astype(np.float64) @ q[0].astype(np.float64))
    w = np.exp(s - s.max())
    ref = (w[:, None] * v[:, 0].astype(np.float64)).sum(0) / w.sum()
    np.testing.assert_allclose(_decode_single(q, k, v, 16, 16, 0.3)[0], ref, atol=1e-12)


def test_gqa_head_mapping_and_context_length():
    """Query head h reads KV head h // G; exactly context_len tokens are read."""
    N, Hq, Hkv, D, B, P = 3, 6, 2, 4, 4, 10
    G = Hq // Hkv
    kc = RNG.standard_normal((P, B, Hkv, D)).astype(np.float32)
    vc = RNG.standard_normal((P, B, Hkv, D)).astype(np.float32)
    bt = np.array([[7, 1, -1], [2, -1, -1], [5, 9, 3]], np.int32)
    ctx = np.array([1, 1, 1], np.int32)
    q = RNG.standard_normal((N, Hq, D)).astype(np.float32)
    o = oracle.decode(q, kc, vc, bt, ctx, 0.5)
    for s in range(N):
        for h in range(Hq):
            np.testing.assert_array_equal(o[s, h], vc[bt[s, 0], 0, h // G].astype(np.float64))
    # equal keys within each sequence: output = mean of exactly ctx values
    kc2 = np.ones_like(kc)
    ctx = np.array([6, 3, 9], np.int32)
    o = oracle.decode(q, kc2, vc, bt, ctx, 0.5)
    for s in range(N):
        rows = [vc[bt[s, j // B], j % B] for j in range(ctx[s])]
        for h in range(Hq):
            want = np.mean([r[h // G] for r in rows], axis=0, dtype=np.float64)
            np.testing.assert_allclose(o[s, h], want, atol=1e-12)


def test_empty_context_is_zero_and_bad_table_rejected():
    kc = np.zeros((2, 4, 1, 2), np.float32)
    q = np.ones((1, 1, 2), np.float32)
    o = oracle.decode(q, kc, kc, np.array([[-1]], np.int32), np.array([0], np.int32), 1.0)
    assert np.all(o == 0)
    with pytest.raises(ValueError):
        oracle.decode(q, kc, kc, np.array([[-1]], np.int32), np.array([1], np.int32), 1.0)
    with pytest.raises(ValueError):
        oracle.decode(q, kc, kc, np.array([[0]], np.int32), np.array([5], np.int32), 1.0)


def test_bf16_widening_exact():
    vals = np.array([1.0, -2.0, 1.5, 0.0, 3.140625, -0.0078125, 65280.0, 1e-3], np.float32)
    bits = _bf16_bits(vals)
    assert bits[:3].tolist() == [0x3F80, 0xC000, 0x3FC0]
    D = vals.shape[0]
    v = bits.reshape(1, 1, D)
    k = np.zeros((1, 1, D), np.uint16)
    q = np.zeros((1, 1, D), np.uint16)
    kp = np.zeros((2, 1, 1, D), np.uint16)
    vp = np.zeros((2, 1, 1, D), np.uint16)
    kp[1] = k
    vp[1] = v
    o = oracle.decode(q, kp, vp, np.array([[1]], np.int32), np.array([1], np.int32), 1.0)
    np.testing.assert_array_equal(o[0, 0], oracle.bf16_bits_to_f64(bits))
    assert o[0, 0, 0] == 1.0 and o[0, 0, 1] == -2.0 and o[0, 0, 2] == 1.5


# --------------------------------------------------------------- prefill
def _prefill_case(seed=0, B=4, Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(seed)
    P = 40
    kc = rng.standard_normal((P, B, Hkv, D)).astype(np.float32)
    vc = rng.standard_normal((P, B, Hkv, D)).astype(np.float32)
    perm = rng.permutation(P)
    bt = np.full((2, 12), -1, np.int32)
    bt[0, :10] = perm[:10]
    bt[1, :6] = perm[10:16]
    ctx = np.array([37, 21], np.int32)
    q_start = np.array([30, 0], np.int32)  # chunk 0: positions 30..36 of seq 0; chunk 1: 0..20 of seq 1
    cu = np.array([0, 7, 28], np.int32)
    q = rng.standard_normal((28, Hq, D)).astype(np.float32)
    return q, cu, q_start, np.array([0, 1], np.int32), kc, vc, bt, ctx


def test_prefill_matches_decode_on_truncated_context():
    q, cu, qs, soc, kc, vc, bt, ctx = _prefill_case()
    o = oracle.prefill(q, cu, qs, soc, kc, vc, bt, ctx, 0.35)
    for c in range(2):
        for i in range(cu[c + 1] - cu[c]):
            p = qs[c] + i
            row = cu[c] + i
            d = oracle.decode(q[row][None], kc, vc, bt[soc[c]][None], np.array([p + 1], np.int32), 0.35)
            np.testing.assert_allclose(o[row], d[0], rtol=0, atol=1e-14)


def test_prefill_first_position_and_causal_limit():
    q, cu, qs, soc, kc, vc, bt, ctx = _prefill_case(seed=1)
    o = oracle.prefill(q, cu, qs, soc, kc, vc, bt, ctx, 0.35)
    G = q.shape[1] // kc.shape[2]
    # chunk 1 starts at position 0: its first query sees only token 0, output = v_0 exactly
    for h in range(q.shape[1]):
        np.testing.assert_array_equal(o[cu[1], h], vc[bt[1, 0], 0, h // G].astype(np.float64))
    # changing K/V of future tokens (positions > p) does not change query p
    kc2, vc2 = kc.copy(), vc.copy()
    B = kc.shape[1]
    for j in range(31, 37):  # seq 0, positions 31..36 (future of query at 30)
        kc2[bt[0, j // B], j % B] += 5.0
        vc2[bt[0, j // B], j % B] -= 3.0
    o2 = oracle.prefill(q, cu, qs, soc, kc2, vc2, bt, ctx, 0.35)
    np.testing.assert_array_equal(o2[0], o[0])
    assert not np.allclose(o2[1], o[1])
    # a chunk that ends beyond the sequence's context is rejected
    with pytest.raises(ValueError):
        oracle.prefill(q, cu, qs, soc, kc, vc, bt, np.array([36, 21], np.int32), 0.35)


# ---- manager-block -> kernel-block remap ("PagedAttention学习笔记", 块表与槽位映射, 混合块)

def test_map_to_kernel_blocks_worked_example():
    # the 40-token sequence of the worked example with 32-token manager blocks 7, 2 (and a padding entry):
    # with 16-token kernel blocks, manager block 7 is kernel blocks 14, 15 and block 2 is 4, 5
    got = oracle.map_to_kernel_blocks(np.array([[7, 2, -1]], np.int32), 2)
    assert got.tolist() == [[14, 15, 4, 5, -1, -1]]


def test_map_to_kernel_blocks_keeps_every_slot():
    """Every position's slot through the manager table (block size ratio*B) equals its slot through the
    kernel table (block size B): the remap changes the bookkeeping, never the address."""
    rng = np.random.default_rng(21)
    for ratio, Bk in ((2, 16), (4, 8), (3, 16), (1, 32)):
        Bm = ratio * Bk
        P = 9
        L = rng.integers(1, 4 * Bm, size=5)
        width = int(-(-L.max() // Bm))
        mgr = np.full((5, width), -1, np.int32)
        for s in range(5):
            nb = -(-int(L[s]) // Bm)
            mgr[s, :nb] = rng.permutation(P)[:nb]
        kern = oracle.map_to_kernel_blocks(mgr, ratio)
        seq = np.repeat(np.arange(5, dtype=np.int32), [int(x) for x in L])
        pos = np.concatenate([np.arange(int(x), dtype=np.int32) for x in L])
        s_mgr, e1 = oracle.slot_mapping(mgr, seq, pos, Bm, P)
        s_ker, e2 = oracle.slot_mapping(kern, seq, pos, Bk, P * ratio)
        assert e1 == e2 == 0
        assert np.array_equal(s_mgr, s_ker)


# ---- fp8 (e4m3) pools: the oracle's format against the format's defining values

def test_e4m3_defining_values():
    assert oracle.e4m3_value(0x00) == 0.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9  # smallest subnormal
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6  # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x3C) == 1.5
    assert oracle.e4m3_value(0x7E) == 448.0  # largest finite
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))  # strictly increasing over the finite codes
    for c in range(0x7F):
        assert oracle.e4m3_value(c | 0x80) == -vals[c] or (c == 0 and np.signbit(oracle.e4m3_value(0x80)))


def test_e4m3_encode_round_trip_ties_and_saturation():
    for c in range(0x7F):
        v = oracle.e4m3_value(c)
        assert oracle.e4m3_encode(v) == c and oracle.e4m3_encode(-v) == (c | 0x80)
    for c in range(0x7E):  # midpoints go to the code with an even mantissa
        mid = (oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)) / 2
        if np.float32(mid) == mid:
            assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1)
    assert oracle.e4m3_encode(449.0) == 0x7E and oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-500.0) == 0xFE
    rng = np.random.default_rng(3)
    finite = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    for x in rng.standard_normal(300).astype(np.float32) * 40:
        got = oracle.e4m3_value(oracle.e4m3_encode(x))
        assert abs(abs(x) - abs(got)) <= np.abs(finite - abs(x)).min() + 1e-12  # a nearest code


def test_fp8_write_round_trips_representable_values():
    """Values that are exactly code * scale come back exactly through the quantising write."""
    import torch
    scale = 0.03125  # a power of two: x * (1 / scale) is exact
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = np.array([oracle.e4m3_value(c) * scale for c in codes], dtype=np.float32)
    bits = torch.from_numpy(vals).to(torch.bfloat16)
    assert torch.equal(bits.float(), torch.from_numpy(vals))  # every value is also a bf16
    knew = bits.view(torch.int16).numpy().view(np.uint16).reshape(1, 1, -1)
    kc = np.zeros((1, 1, 1, knew.shape[2]), np.uint8)
    vc = np.zeros_like(kc)
    assert oracle.write_kv_fp8(knew, knew, kc, vc, np.array([0]), scale, scale) == 0
    assert np.array_equal(kc.reshape(-1), codes)
    assert np.array_equal(oracle.dequant_e4m3(kc, scale).reshape(-1), vals.astype(np.float64))


def test_fp8_write_reciprocal_rounding_at_non_power_of_two_scales():
    """The quantising write's reading: code = e4m3(x * (1/scale)) with the reciprocal and the product each
    rounded to float ("KV cache 显存管理…", KV size formula leaves the element format open; the reading is the
    one stated for the fp8 pools).  Each case below is a bf16 value whose float product lands exactly on the
    midpoint between two codes, or just off it, while a plausible slip lands on the other side:

    * scale 0.37f: 1/0.37f rounds to 2.702702760696411 (0x402CF915); 0.2890625 * that = 0.78125000168 in exact
      arithmetic, which rounds in float to 0.78125, the midpoint of 0.75 (0x34) and 0.8125 (0x35): the tie goes
      to the even code 0x34.  Keeping the product in double would give 0x35.
    * scale 0.7f: 1/0.7f = 1.4285714626312256; 0.2734375 * that rounds to 0.390625, the midpoint of 0.375 (0x2C)
      and 0.40625 (0x2D): 0x2C.  Dividing by the scale in double (0.39062500665) would give 0x2D.
    * scale 0.9f: 1/0.9f = 1.1111111640930176; 0.3515625 * that rounds to 0.39062503 (above the same midpoint):
      0x2D.  Dividing by the scale in float gives exactly 0.390625, hence 0x2C.
    * scale 0.6f: 1/0.6f = 1.6666666269302368; 0.0087890625 * that rounds to 0.0146484375, the midpoint of the
      largest subnormal 7 * 2^-9 (0x07) and the smallest normal 2^-6 (0x08): the even code 0x08.  Division in
      double or float, or the product in double, all fall below the midpoint: 0x07.
    Negated inputs give the same codes with the sign bit set."""
    import torch
    cases = [(0.37, 0.2890625, 0x34), (0.7, 0.2734375, 0x2C), (0.9, 0.3515625, 0x2D), (0.6, 0.0087890625, 0x08)]
    for scale, x, code in cases:
        vals = torch.tensor([x, -x], dtype=torch.float32)
        bits = vals.to(torch.bfloat16)
        assert torch.equal(bits.float(), vals)  # the inputs are exact bf16 values
        knew = bits.view(torch.int16).numpy().view(np.uint16).reshape(1, 1, 2)
        vnew = np.zeros_like(knew)
        kc = np.zeros((1, 1, 1, 2), np.uint8)
        vc = np.zeros_like(kc)
        assert oracle.write_kv_fp8(knew, vnew, kc, vc, np.array([0]), scale, 1.0) == 0
        assert kc.reshape(-1).tolist() == [code, code | 0x80], (scale, x, kc.reshape(-1).tolist())
        # the same value through the V pool's scale
        kc[:] = 0
        vc[:] = 0
        assert oracle.write_kv_fp8(vnew, knew, kc, vc, np.array([0]), 1.0, scale) == 0
        assert vc.reshape(-1).tolist() == [code, code | 0x80]


# ---- sharing ("什么是 PagedAttention？", 共享但不污染状态): sequences that map the same physical prefix blocks

def _shared_batch(seed, B=16, Hq=8, Hkv=2, D=32):
    """Four sequences over one pool.  Sequences 0 and 1 share physical prefix blocks 5, 9, 2 and each has a
    private tail block (7 and 11); block 11 is filled with a copy of block 7, so their K/V are equal token by
    token.  Sequence 2 shares the prefix but its tail block 13 holds different values.  Sequence 3 holds the
    same K/V as sequence 0 in entirely different physical blocks (a copy of the prefix in 20, 21, 22 and of the
    tail in 23)."""
    rng = np.random.default_rng(seed)
    P = 24
    kc = rng.standard_normal((P, B, Hkv, D)).astype(np.float32)
    vc = rng.standard_normal((P, B, Hkv, D)).astype(np.float32)
    for dst, src in ((11, 7), (20, 5), (21, 9), (22, 2), (23, 7)):
        kc[dst] = kc[src]
        vc[dst] = vc[src]
    bt = np.array([[5, 9, 2, 7], [5, 9, 2, 11], [5, 9, 2, 13], [20, 21, 22, 23]], np.int32)
    L = 3 * B + 5
    ctx = np.full(4, L, np.int32)
    q1 = rng.standard_normal((Hq, D)).astype(np.float32)
    q = np.stack([q1, q1, q1, q1])
    return q, kc, vc, bt, ctx


def test_shared_prefix_sequences_give_identical_outputs():
    """Two sequences of one batch whose tables map the same physical prefix blocks, with equal tails and
    equal queries, give bitwise-equal outputs; a sequence with the same prefix but a different tail does not;
    the same K/V at another placement gives the same outputs (paged == contiguous)."""
    q, kc, vc, bt, ctx = _shared_batch(5)
    for threads in (1, 4):
        o = oracle.decode(q, kc, vc, bt, ctx, 0.2, num_threads=threads)
        assert np.array_equal(o[0], o[1])
        assert np.array_equal(o[0], o[3])
        assert not np.allclose(o[0], o[2], atol=1e-6)
    # with the queries of sequence 1 changed the outputs differ (the rows are not read from one sequence)
    q2 = q.copy()
    q2[1] = -q2[1]
    o2 = oracle.decode(q2, kc, vc, bt, ctx, 0.2)
    assert np.array_equal(o2[0], o[0]) and not np.allclose(o2[1], o2[0], atol=1e-6)
    # a shorter context on sequence 1 that stops inside the shared prefix reads only shared blocks: it equals
    # the same length on sequence 2, whose different tail is then never read
    ctx2 = ctx.copy()
    ctx2[1] = ctx2[2] = 2 * kc.shape[1] + 3
    o3 = oracle.decode(q, kc, vc, bt, ctx2, 0.2)
    assert np.array_equal(o3[1], o3[2])


def test_shared_prefix_prefill_identical_for_identical_chunks():
    """The same sharing for prefill chunks: chunks of two sequences that share their prefix blocks and have
    equal tails, with equal queries at equal positions, give bitwise-equal outputs."""
    q, kc, vc, bt, ctx = _shared_batch(6)
    n = 9
    rng = np.random.default_rng(7)
    qc = rng.standard_normal((n, q.shape[1], q.shape[2])).astype(np.float32)
    qp = np.concatenate([qc, qc, qc])
    cu = np.array([0, n, 2 * n, 3 * n], np.int32)
    start = np.full(3, int(ctx[0]) - n, np.int32)
    o = oracle.prefill(qp, cu, start, np.array([0, 1, 2], np.int32), kc, vc, bt, ctx, 0.2)
    assert np.array_equal(o[:n], o[n:2 * n])
    assert not np.allclose(o[:n], o[2 * n:], atol=1e-6)


# ---- the float64 input branch (used for e4m3 pools read back as code * scale)

def test_float64_inputs_equal_the_same_values_as_float32():
    """Decode and prefill on float64 arrays holding float32 values give exactly the float32 results: the
    widening is exact and the arithmetic is fp64 either way.  Guards the float64 element loads and sizes."""
    q, cu, qs, soc, kc, vc, bt, ctx = _prefill_case(seed=3)
    o32 = oracle.prefill(q, cu, qs, soc, kc, vc, bt, ctx, 0.35)
    o64 = oracle.prefill(q.astype(np.float64), cu, qs, soc, kc.astype(np.float64), vc.astype(np.float64), bt, ctx,
                         0.35)
    assert np.array_equal(o32, o64)
    qd = q[:2]
    d32 = oracle.decode(qd, kc, vc, bt, ctx, 0.35)
    d64 = oracle.decode(qd.astype(np.float64), kc.astype(np.float64), vc.astype(np.float64), bt, ctx, 0.35)
    assert np.array_equal(d32, d64)
    # values that float32 cannot hold are used as they are: a float64 pool with a 1e-12 offset on one key
    # changes the scores (a float32 load of the same memory would not see it)
    kc64 = kc.astype(np.float64)
    kc64[bt[0, 0], 0, 0, 0] += 1e-12 * 2 ** 20
    d64b = oracle.decode(qd.astype(np.float64), kc64, vc.astype(np.float64), bt, ctx, 0.35)
    assert not np.array_equal(d64b[0], d32[0])
