"""Pins of the CPU oracle to things other than itself: the values the pages
print for their worked examples (``tests/golden/``), closed forms, library
routines for the special cases that reduce to them, brute force on tiny inputs
and invariants.  Each pin is a function taking the oracle routine under test,
so the mutation tests at the end can show that a plausible mistake planted in
the oracle (on the CPU) fails it.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_grouped_topk_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


TRACED = golden("traced_scenario.json")
GEMM = golden("gemm_unit_example.json")


# ---------------------------------------------------------------------------
# e4m3 and bf16 codecs
# ---------------------------------------------------------------------------

def test_e4m3_table_closed_forms():
    d = O.e4m3_decode
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0       # 1.75 * 2**8
    assert d(0x01) == 2.0 ** -9                          # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9                      # largest subnormal
    assert d(0x08) == 2.0 ** -6                          # smallest normal
    assert d(0x38) == 1.0                                # exponent field 7 = bias
    assert d(0x3C) == 1.5
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x80) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    assert len(set(float(d(c)) for c in finite)) == 253  # +0 and -0 compare equal


def pin_encode_roundtrip(encode):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    vals[codes == 0x80] = -0.0
    assert np.array_equal(encode(vals), codes)


def pin_encode_nearest_even(encode):
    """Brute force against the definition: the nearest finite code, ties to the
    even mantissa, saturating beyond 448."""
    rng = np.random.default_rng(1)
    pos = np.array([c for c in range(0x7F)], dtype=np.uint8)       # +0 .. 448
    pv = O.e4m3_decode(pos)
    ties = (pv[1:] + pv[:-1]) / 2                                   # every midpoint
    v = np.concatenate([rng.uniform(-500, 500, 4000), rng.uniform(-0.05, 0.05, 4000),
                        rng.uniform(-3e-3, 3e-3, 2000), ties, -ties]).astype(np.float32)
    got = encode(v)
    for x, c in zip(v, got):
        a = abs(float(x))
        if a >= 448.0:
            want = 0x7E
        else:
            dist = np.abs(pv - a)
            best = np.flatnonzero(dist == dist.min())
            want = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        if x < 0 or (x == 0 and math.copysign(1.0, float(x)) < 0):
            want |= 0x80
        assert int(c) == want, (float(x), int(c), want)


def test_e4m3_encode_roundtrip():
    pin_encode_roundtrip(O.e4m3_encode)


def test_e4m3_encode_nearest_even():
    pin_encode_nearest_even(O.e4m3_encode)


def test_e4m3_encode_matches_torch_cast():
    """PyTorch's fp32 -> float8_e4m3fn cast is round-to-nearest-even; it agrees
    with the encoder wherever it does not overflow (|v| < 464)."""
    rng = np.random.default_rng(2)
    codes = np.arange(0x7E, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)          # every tie
    v = np.concatenate([mids, -mids, rng.standard_normal(1 << 20).astype(np.float32) * 50,
                        rng.uniform(-463.9, 463.9, 1 << 18).astype(np.float32),
                        rng.uniform(-1e-2, 1e-2, 1 << 18).astype(np.float32)])
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v), want)
    assert O.e4m3_encode(np.float32([1000.0, -470.0]))[0] == 0x7E   # satfinite
    assert O.e4m3_encode(np.float32([1000.0, -470.0]))[1] == 0xFE


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    base = rng.standard_normal(1 << 18).astype(np.float32)
    ties = (base.view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    v = np.concatenate([base, ties.view(np.float32), np.float32([0.0, -0.0, 3.0e38])])
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(v), want)
    assert np.array_equal(O.bf16_bits_to_f32(want), torch.from_numpy(v).to(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------------------
# Per-token FP8 quantisation rule
# ---------------------------------------------------------------------------

def pin_quant_special_cases(quant):
    # a constant group maps every element to 448 with scale c / 448
    c = np.float32(3.25)
    codes, sc = quant(np.full((1, 128), c, np.float32))
    assert np.all(codes == 0x7E) and sc[0, 0] == np.float32(c / np.float32(448.0))
    # an all-zero group takes the 1e-4 floor: codes 0, scale 1e-4 / 448
    codes, sc = quant(np.zeros((1, 256), np.float32))
    assert np.all(codes == 0) and np.all(sc == np.float32(1e-4) / np.float32(448.0))
    # the group's largest magnitude always lands on +-448
    rng = np.random.default_rng(4)
    v = rng.standard_normal((64, 512)).astype(np.float32)
    codes, sc = quant(v)
    g = v.reshape(64, 4, 128)
    arg = np.abs(g).argmax(axis=2)
    top = np.take_along_axis(codes.reshape(64, 4, 128), arg[..., None], axis=2)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))
    # dequantised values are within half an e4m3 step: relative 2**-4 for normals
    deq = O.e4m3_decode(codes).reshape(64, 4, 128) * sc[..., None]
    big = np.abs(g) >= (2.0 ** -6) * sc[..., None]
    assert np.all(np.abs(deq - g)[big] <= np.abs(g)[big] * 2.0 ** -4 + 1e-12)
    # rows are independent: quantising a row alone gives the same bytes
    c1, s1 = quant(v[7:8])
    assert np.array_equal(c1, codes[7:8]) and np.array_equal(s1, sc[7:8])


def test_quant_rule_pins():
    pin_quant_special_cases(O.quantize_rows)


def test_quant_scale_is_fp32_rule():
    """The scale is amax/448 and the multiplier 448/amax, both fp32 divisions
    (DeepEP notes §11); checked against Python's correctly rounded double
    division narrowed to fp32 (exact for a single fp32 division)."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((16, 128)) * rng.uniform(1e-3, 1e3, (16, 1))).astype(np.float32)
    _, sc = O.quantize_rows(v)
    for r in range(16):
        amax = float(np.max(np.abs(v[r])))
        assert sc[r, 0] == np.float32(amax / 448.0)


# ---------------------------------------------------------------------------
# Routing
# ---------------------------------------------------------------------------

def traced_ids(swap=False):
    idx, w = W.traced_routes(seed=0, swap_token_21=swap)
    return idx.numpy(), w.numpy()


def pin_traced_counts(route_fn):
    idx, _ = traced_ids()
    rr = route_fn(idx, 8, 128)
    assert rr.counts.tolist() == TRACED["counts"]["global"]
    assert rr.counts[:2].tolist() == TRACED["counts"]["rank0"]
    assert int(rr.counts.sum()) == TRACED["total_routes"]["value"] == 112 * 2
    # token (2, 5) = global 21 is the only route of E1 and of E6: row 0 of each
    t21 = 16 + 5
    assert rr.src_map[t21].tolist() == [1 * 128 + 0, 6 * 128 + 0]
    # with the pages' own capacity M = W*C = 256, E1's row is q = 256
    rr256 = route_fn(idx, 8, TRACED["flat_row_e1"]["M"])
    assert int(rr256.src_map[t21, 0]) == TRACED["flat_row_e1"]["q"] != TRACED["flat_row_e1"]["not"]
    # E0 on rank 0 receives 16 / 31 / 64 routes from source ranks 1 / 2 / 3
    src = W.source_rank_of_tokens(W.WORKLOADS["traced"]).numpy()
    per_src = [int(((idx[:, 0] == 0) & (src == r)).sum()) for r in (1, 2, 3)]
    assert per_src == TRACED["rank0_e0_sources"]["value"]


def test_traced_routing_pins():
    pin_traced_counts(O.route)


def test_replay_counts():
    idx, _ = traced_ids(swap=True)
    rr = O.route(idx, 8, 128)
    assert [int(rr.counts[e]) for e in TRACED["replay"]["experts"]] == TRACED["replay"]["after"]
    idx0, _ = traced_ids(swap=False)
    rr0 = O.route(idx0, 8, 128)
    assert [int(rr0.counts[e]) for e in TRACED["replay"]["experts"]] == TRACED["replay"]["before"]


def pin_source_slots_traced(fn):
    """The per-source fixed-slot layout ("DeepEP 架构与实现笔记", §9.5) on the
    traced scenario with the pages' own per-rank slot count C = 64 (W = 4, so
    each expert holds W*C = 256 rows): E0 receives 16, 31 and 64 routes from
    source ranks 1, 2 and 3 ("SGLang、NCCL 与 MoE EP", §2.3.7), each group in
    its own source's 64-row range; masked_m equals the global counts."""
    idx, _ = traced_ids()
    src = W.source_rank_of_tokens(W.WORKLOADS["traced"]).numpy()
    C = TRACED["flat_row_e1"]["M"] // 4
    res = fn(idx, 8, 2, C, src)
    assert res.seg_counts[0].tolist() == [0] + TRACED["rank0_e0_sources"]["value"]
    assert res.seg_counts[7].tolist() == [0] + TRACED["rank0_e0_sources"]["value"]
    assert res.seg_counts[1].tolist() == [0, 0, 1, 0] == res.seg_counts[6].tolist()
    assert res.counts.tolist() == TRACED["counts"]["global"]
    # token (2, 5) = global 21: source rank 2's first slot of E1 and of E6
    M = 4 * C
    assert res.src_map[16 + 5].tolist() == [1 * M + 2 * C, 6 * M + 2 * C]
    # the first token of rank 3 (global 48) opens rank 3's range of E0 and E7
    assert res.src_map[48].tolist() == [0 * M + 3 * C, 7 * M + 3 * C]
    assert res.dropped == 0 and not res.bad_id


def test_source_slot_layout_pins():
    pin_source_slots_traced(O.route_source_slots)


def test_source_slot_layout_invariants():
    """Every route sits in its source's fixed range of its expert; read in row
    order, an expert's valid rows list the same routes as the canonical padded
    layout (sources are concatenated in token order); a source with more
    routes to one expert than its range holds drops the later ones."""
    rng = np.random.default_rng(12)
    E, L, K, T = 16, 4, 3, 90
    W_ = E // L
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int64)
    idx[rng.random((T, K)) < 0.1] = -1
    src = np.minimum(np.arange(T) // -(-T // W_), W_ - 1)
    mt = 40
    res = O.route_source_slots(idx, E, L, mt, src)
    R = W_ * mt
    canon = O.route(idx, E, R)
    assert res.dropped == 0 and canon.dropped == 0
    assert res.counts.tolist() == canon.counts.tolist()
    for e in range(E):
        rows = {}
        for t, k in np.argwhere(res.src_map // R == e):
            q = int(res.src_map[t, k]) - e * R
            r, p = divmod(q, mt)
            assert r == src[t] and p < res.seg_counts[e, r]
            rows[q] = (t, k)
        in_row_order = [rows[q] for q in sorted(rows)]
        by_slot = sorted((int(canon.src_map[t, k]), (t, k)) for t, k in np.argwhere(canon.src_map // R == e))
        assert in_row_order == [tk for _, tk in by_slot]
    small = O.route_source_slots(idx, E, L, 2, src)
    assert small.dropped == int(np.maximum(res.seg_counts - 2, 0).sum())
    assert small.seg_counts.max() <= 2


def test_placement_and_byte_accounting():
    p = TRACED["placement"]
    for g, r, l in p["routes"]:
        assert O.expert_placement(g, p["L"]) == (r, l)
    idx, _ = traced_ids()
    src = W.source_rank_of_tokens(W.WORKLOADS["traced"]).numpy()
    st = O.route_stats(idx, 2, src)
    b = TRACED["bytes"]
    assert st["routes"] == b["routes"] and st["messages"] == b["routes"]
    assert st["cross_rank_routes"] == b["cross_rank_routes"]
    assert st["routes"] * b["H"] * 2 == b["route_bytes"] == int(1.75 * 2 ** 20)
    assert st["cross_rank_routes"] * b["H"] * 2 == b["cross_rank_bytes"] == int(1.25 * 2 ** 20)


def pin_route_canonical(route_fn):
    """Independent restatement of the canonical order with a library stable
    sort: the slot of route i in expert e is its position among e's routes
    sorted by route id; brute force over many small random cases, with -1
    padding and capacity overflow."""
    rng = np.random.default_rng(6)
    for trial in range(300):
        E = int(rng.integers(1, 9))
        K = int(rng.integers(1, min(E, 4) + 1))
        T = int(rng.integers(0, 40))
        R = int(rng.integers(1, 12))
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)
        rr = route_fn(idx, E, R)
        flat = idx.reshape(-1)
        valid = np.flatnonzero(flat >= 0)
        order = valid[np.argsort(flat[valid], kind="stable")]
        want = np.full(T * K, -1, np.int64)
        slot_of = {}
        for i in order:
            e = int(flat[i])
            s = slot_of.get(e, 0)
            slot_of[e] = s + 1
            if s < R:
                want[i] = e * R + s
        assert np.array_equal(rr.src_map.reshape(-1), want)
        n = np.bincount(flat[valid], minlength=E) if len(valid) else np.zeros(E, int)
        assert np.array_equal(rr.counts, np.minimum(n, R))
        assert rr.dropped == int(np.maximum(n - R, 0).sum())
        assert int(rr.counts.sum()) + rr.dropped == len(valid)
        # bijection of the kept routes onto each expert's valid prefix
        for e in range(E):
            rows = sorted(int(q) - e * R for q in rr.src_map.reshape(-1) if q >= 0 and q // R == e)
            assert rows == list(range(int(rr.counts[e])))


def test_route_canonical_order():
    pin_route_canonical(O.route)


def test_route_bad_id_and_padding():
    idx = np.array([[0, -1], [5, 1], [-3, 0]], np.int64)
    rr = O.route(idx, 4, 8)
    assert rr.bad_id
    assert rr.src_map.tolist() == [[0, -1], [-1, 8], [-1, 1]]
    assert rr.counts.tolist() == [2, 1, 0, 0]
    rr = O.route(np.zeros((0, 3), np.int64), 4, 8)        # empty rank
    assert rr.counts.tolist() == [0, 0, 0, 0] and rr.src_map.shape == (0, 3)


def test_scatter_places_rows():
    x = np.arange(12, dtype=np.float32).reshape(3, 4)
    idx = np.array([[1, 0], [1, -1], [0, 1]], np.int64)
    rr = O.route(idx, 2, 4)
    recv = O.scatter(x, rr.src_map, 2, 4)
    assert np.array_equal(recv[1, 0], x[0]) and np.array_equal(recv[1, 1], x[1])
    assert np.array_equal(recv[1, 2], x[2]) and np.array_equal(recv[0, 0], x[0])
    assert np.array_equal(recv[0, 1], x[2]) and np.all(np.isnan(recv[0, 2:]))


# ---------------------------------------------------------------------------
# Expert math
# ---------------------------------------------------------------------------

def _codes(vals):
    return O.e4m3_encode(np.asarray(vals, np.float32))


def pin_expert_hand_example(forward):
    """H = I = 128, one row, unit scales.  x = e0 + 2*e1; gate row 0 picks
    x[0] (= 1), up row 0 picks 0.5*x[1] (= 1), so Z[0] = SiLU(1)*1 = sigma(1)
    and every other Z is 0.  Z requantises to code 448 with scale sigma(1)/448,
    and the down row h has weight (h % 5 - 2) on Z[0], so
    out[h] = (h % 5 - 2) * sigma(1) (up to the fp32 rounding of the scale).
    Gate row 3 reads x[1] through column 1 to catch a transposed operand."""
    H = I = 128
    x = np.zeros((1, H), np.float32)
    x[0, 0], x[0, 1] = 1.0, 2.0
    xq = _codes(x)
    sx = np.ones((1, 1), np.float32)
    w13 = np.zeros((2 * I, H), np.float32)
    w13[0, 0] = 1.0
    w13[I + 0, 1] = 0.5
    w13[3, 1] = 2.0          # gate 3 = 4, up 3 = 0 -> Z[3] = 0
    w13[I + 5, 1] = 1.0      # up 5 = 2, gate 5 = 0 -> Z[5] = 0
    w2 = np.zeros((H, I), np.float32)
    w2[:, 0] = np.arange(H) % 5 - 2
    out, zq, sz, G = forward(xq, sx, _codes(w13), np.ones((2, 1), np.float32), _codes(w2), np.ones((1, 1), np.float32))
    sig1 = 1.0 / (1.0 + math.exp(-1.0))
    assert G[0, 0] == 1.0 and G[0, I] == 1.0 and G[0, 3] == 4.0 and G[0, I + 5] == 2.0
    assert zq[0, 0] == 0x7E and np.all(zq[0, 1:] == 0)
    assert sz[0, 0] == np.float32(np.float32(sig1) / np.float32(448.0))
    want = (np.arange(H) % 5 - 2) * sig1
    assert np.allclose(out[0], want, rtol=1e-6, atol=0)


def test_expert_hand_example():
    pin_expert_hand_example(O.expert_forward)


def pin_gemm_integer_case(gemm):
    """All scales powers of two and all operands small integers exact in e4m3:
    the block-scaled GEMM is an exact integer matmul (numpy int64) times the
    scale product."""
    rng = np.random.default_rng(7)
    m, N, K = 5, 256, 384
    a = rng.integers(-8, 9, (m, K)).astype(np.float32)
    w = rng.integers(-8, 9, (N, K)).astype(np.float32)
    sa = np.float32(2.0) ** rng.integers(-3, 4, (m, K // 128)).astype(np.float32)
    sw = np.float32(2.0) ** rng.integers(-3, 4, (N // 128, K // 128)).astype(np.float32)
    got = gemm(_codes(a), sa, _codes(w), sw)
    ai, wi = a.astype(np.int64), w.astype(np.int64)
    want = np.zeros((m, N))
    for g in range(K // 128):
        part = ai[:, g * 128:(g + 1) * 128] @ wi[:, g * 128:(g + 1) * 128].T
        want += sa[:, g][:, None].astype(np.float64) * np.repeat(sw[:, g], 128)[None, :] * part
    assert np.array_equal(got, want)


def test_gemm_integer_case():
    pin_gemm_integer_case(O.gemm_block_scaled)


def pin_gemm_brute_force(gemm):
    """Triple loop straight from the block-scale formula, two rows."""
    rng = np.random.default_rng(8)
    m, N, K = 2, 128, 256
    aq = rng.integers(0, 0x7E, (m, K)).astype(np.uint8) | (rng.integers(0, 2, (m, K)) * 0x80).astype(np.uint8)
    wq = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    sa = rng.uniform(0.5, 2, (m, 2)).astype(np.float32)
    sw = rng.uniform(0.5, 2, (1, 2)).astype(np.float32)
    got = gemm(aq, sa, wq, sw)
    A, Wd = O.e4m3_decode(aq), O.e4m3_decode(wq)
    for i in range(m):
        for n in (0, 1, 77, 127):
            tot = 0.0
            for g in range(2):
                s = 0.0
                for k in range(g * 128, g * 128 + 128):
                    s += A[i, k] * Wd[n, k]
                tot += float(sa[i, g]) * float(sw[n // 128, g]) * s
            assert abs(got[i, n] - tot) <= 1e-9 * max(1.0, abs(tot))


def test_gemm_brute_force():
    pin_gemm_brute_force(O.gemm_block_scaled)


def test_silu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 40.0, -800.0])
    s = O.silu(g)
    assert s[0] == 0.0
    assert abs(s[1] - 1 / (1 + math.exp(-1))) < 1e-15
    assert abs(s[2] + 1 / (1 + math.exp(1))) < 1e-15
    assert abs(s[3] - 40.0) < 1e-12 and s[4] == 0.0


# ---------------------------------------------------------------------------
# Combine
# ---------------------------------------------------------------------------

def pin_combine_traced(combine):
    ex = TRACED["combine_example"]
    out = np.zeros((4, 3), np.float32)
    out[1, 0], out[2, 0] = ex["outputs"]
    src = np.array([[1, 2]], np.int32)
    w = np.array([ex["weights"]], np.float32)
    y = combine(out, src, w)
    assert y[0, 0] == ex["value"] and y[0, 1] == 0.0


def test_combine_traced_example():
    pin_combine_traced(O.combine_fp64)
    pin_combine_traced(O.combine_f32_sequential)


def test_combine_identity_experts_return_input():
    """Identity experts (out = recv) with weights summing to 1 give y == x
    bitwise after the BF16 rounding."""
    idx, w = traced_ids()
    x = W.activations(112, 256, 3).float().numpy()
    rr = O.route(idx, 8, 128)
    recv = O.scatter(x, rr.src_map, 8, 128).reshape(8 * 128, 256)
    y32 = O.combine_f32_sequential(recv, rr.src_map, w)
    assert np.array_equal(y32, x)
    y64 = O.combine_fp64(recv, rr.src_map, w)
    assert np.array_equal(O.f32_to_bf16_rne(y64.astype(np.float32)), x)


# A two-route token whose products nearly cancel: the fp32 rounding of each
# product is then as large as the sum itself, so the three plausible readings
# of "fp32 accumulation" -- product and sum each rounded, a fused multiply-add
# for the second term, or fp64 accumulation rounded once -- land on three
# different BF16 values.  Inputs as bit patterns: router weights fp32, expert
# outputs BF16 (the dtype the combine reads).
COMBINE_ROUNDING = {"w_bits": [0x3EE87226, 0x3EDA5BAF], "v_bits": [0x3F78, 0xBF84]}


def _f32_round(x: Fraction) -> Fraction:
    """Nearest fp32 to an exactly representable-in-double rational (ties to
    even): ``struct`` packs a double into binary32 with IEEE rounding."""
    d = float(x)
    assert Fraction(d) == x, "value not exact in fp64"
    return Fraction(struct.unpack("<f", struct.pack("<f", d))[0])


def _bf16_round(x: Fraction) -> float:
    """Nearest BF16 (ties to even) of an exact rational, by exact arithmetic."""
    if x == 0:
        return 0.0
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > abs(x):
        e -= 1
    while Fraction(2) ** (e + 1) <= abs(x):
        e += 1
    q = Fraction(2) ** (e - 7)                     # 8 significant bits
    n = abs(x) / q
    f = math.floor(n)
    r = n - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return float((1 if x > 0 else -1) * f * q)


def _combine_rounding_readings():
    w = [Fraction(struct.unpack("<f", struct.pack("<I", b))[0]) for b in COMBINE_ROUNDING["w_bits"]]
    v = [Fraction(struct.unpack("<f", struct.pack("<I", b << 16))[0]) for b in COMBINE_ROUNDING["v_bits"]]
    p0 = _f32_round(w[0] * v[0])
    two = _f32_round(p0 + _f32_round(w[1] * v[1]))     # product and sum each rounded
    fused = _f32_round(p0 + w[1] * v[1])               # fma for the second term
    wide = w[0] * v[0] + w[1] * v[1]                   # fp64 (exact here), rounded once
    return w, v, {"mul_add": _bf16_round(two), "fma": _bf16_round(fused), "fp64": _bf16_round(wide)}


def pin_combine_rounding(combine):
    """The combine's rounding sequence (fp32, product and sum each rounded,
    ascending k from 0, one BF16 rounding at the end), checked on a case where
    the other readings give other results."""
    w, v, want = _combine_rounding_readings()
    out = np.array([[float(v[0]), 0.0], [float(v[1]), 0.0]], np.float32)
    src = np.array([[0, 1]], np.int32)
    ww = np.array([[float(w[0]), float(w[1])]], np.float32)
    y = combine(out, src, ww)
    assert y[0, 0] == want["mul_add"] and y[0, 1] == 0.0


def test_combine_rounding_sequence():
    """"SGLang、NCCL 与 MoE EP", §3.2: each route's output is multiplied by its
    weight once and summed into the token's row; the accumulation is fp32 in
    ascending k (the reading taken here, as the pages do not fix the
    rounding).  The three readings differ on this case, so the pin tells them
    apart; the fp64 oracle combine agrees with the fp64 reading."""
    _, _, want = _combine_rounding_readings()
    assert len({want["mul_add"], want["fma"], want["fp64"]}) == 3
    pin_combine_rounding(O.combine_f32_sequential)
    w, v, _ = _combine_rounding_readings()
    y64 = O.combine_fp64(np.array([[float(v[0])], [float(v[1])]], np.float32), np.array([[0, 1]], np.int32),
                         np.array([[float(w[0]), float(w[1])]], np.float32))
    assert float(O.f32_to_bf16_rne(y64.astype(np.float32))[0, 0]) == want["fp64"]


def test_combine_empty_rank():
    y = O.combine_f32_sequential(np.zeros((8, 16), np.float32), np.zeros((0, 2), np.int32), np.zeros((0, 2), np.float32))
    assert y.shape == (0, 16)


def test_combine_50_arrival_orders():
    """Any bijection of each expert's routes onto its valid prefix is a valid
    dispatch; slot -> map -> combine gives the same y under 50 random arrival
    orders (the CPU check of "SGLang、NCCL 与 MoE EP", appendix B.4)."""
    rng = np.random.default_rng(9)
    idx, w = traced_ids()
    x = W.activations(112, 256, 4).float().numpy()
    rr = O.route(idx, 8, 128)
    E, R = 8, 128
    fexp = rng.standard_normal((E, 256)).astype(np.float32)     # stand-in expert: add a per-expert row
    base = None
    for _ in range(50):
        perm_map = np.full_like(rr.src_map, -1)
        for e in range(E):
            tk = np.argwhere((rr.src_map >= 0) & (rr.src_map // R == e))
            slots = rng.permutation(len(tk))
            for (t, k), s in zip(tk, slots):
                perm_map[t, k] = e * R + s
        recv = O.scatter(x, perm_map, E, R).reshape(E * R, 256)
        out = recv + np.repeat(fexp, R, axis=0)
        y = O.combine_f32_sequential(out, perm_map, w)
        if base is None:
            base = y
        assert np.array_equal(y, base)


# ---------------------------------------------------------------------------
# Tiles and addressing of the [70, 12] example
# ---------------------------------------------------------------------------

def test_gemm_unit_tiles_and_bm_table():
    t = GEMM["tiles"]
    counts = GEMM["shapes"]["counts"]
    assert O.valid_tiles(counts, t["BM"], t["BN"], t["N"]) == t["value"]
    S = GEMM["shapes"]["L"] * GEMM["shapes"]["R"]
    for BM, blocks, covered, fill, Q, grid in GEMM["bm_table"]["rows"]:
        assert O.m_blocks(counts, BM) == blocks
        assert BM * O.m_blocks(counts, BM) == covered
        assert round(100 * O.m_fill_rate(counts, BM), 1) == fill
        assert O.align_index_capacity(S, 2, BM) == Q
        assert O.align_grid(S, 2, BM, 128, 256) == grid
    sp = GEMM["split"]
    both = 2 * O.m_blocks(sp["half"], 64)
    assert both == sp["m_blocks"] and 64 * both == sp["covered"]
    assert round(100 * sum(counts) / (64 * both), 1) == sp["fill_pct"]


def test_gemm_unit_addresses():
    for it in GEMM["addresses"]["items"]:
        assert O.row_major_offset(it["shape"], it["index"]) == it["offset"], it["name"]
    R = GEMM["flat_rows"]["R"]
    for q, e, s in GEMM["flat_rows"]["items"]:
        assert divmod(q, R) == (e, s)


def test_expert_forward_layout_matches_addresses():
    """The oracle's GEMM reads W13 as [E, N, K] (output-major): entry
    W13[0,129,130] multiplies A[65,130] into gateup[65,129]."""
    rng = np.random.default_rng(10)
    aq = np.zeros((128, 256), np.uint8)
    wq = np.zeros((256, 256), np.uint8)
    aq[65, 130] = 0x38                 # 1.0
    wq[129, 130] = 0x40                # 2.0
    wq[130, 129] = 0x48                # 4.0 -- the transposed position
    G = O.gemm_block_scaled(aq, np.ones((128, 2), np.float32), wq, np.ones((2, 2), np.float32))
    assert G[65, 129] == 2.0 and np.count_nonzero(G) == 1


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------

def test_moe_layer_traced_structure():
    """Whole-layer oracle on the traced scenario: the token-21 row is the
    0.25 / 0.75 mix of E1 and E6 applied to the same quantised row."""
    d = W.make_layer_inputs("traced", seed=0)
    x = d["x"].float().numpy()
    y, rr, route_out = O.moe_layer(x, d["topk_idx"].numpy(), d["topk_w"].numpy(), d["w13"].numpy(),
                                   d["s13"].numpy(), d["w2"].numpy(), d["s2"].numpy(), 8, 128)
    xq, sx = O.quantize_rows(x[21:22])
    f1 = O.expert_forward(xq, sx, d["w13"][1].numpy(), d["s13"][1].numpy(), d["w2"][1].numpy(), d["s2"][1].numpy())[0]
    f6 = O.expert_forward(xq, sx, d["w13"][6].numpy(), d["s13"][6].numpy(), d["w2"][6].numpy(), d["s2"][6].numpy())[0]
    assert np.allclose(y[21], 0.25 * f1[0] + 0.75 * f6[0], rtol=1e-12, atol=1e-12)
    assert rr.counts.tolist() == TRACED["counts"]["global"]
    assert np.all(route_out[rr.src_map < 0] == 0)


# ---------------------------------------------------------------------------
# Mutation tests: a plausible mistake planted in the oracle fails a pin
# ---------------------------------------------------------------------------

def _fails(pin, fn):
    try:
        pin(fn)
    except AssertionError:
        return True
    return False


def test_mutants_are_caught():
    # transposed weight operand
    def gemm_t(aq, sa, wq, sw):
        return O.gemm_block_scaled(aq, sa, np.ascontiguousarray(wq.T) if wq.shape[0] == wq.shape[1] else wq[:, ::-1], sw)
    assert _fails(pin_gemm_integer_case, gemm_t)

    # weight scale of the wrong block (n % 128 instead of n // 128) -> dropped term
    def gemm_noscale(aq, sa, wq, sw):
        return O.gemm_block_scaled(aq, sa, wq, np.ones_like(sw))
    assert _fails(pin_gemm_integer_case, gemm_noscale)

    # gate and up swapped
    def fwd_swapped(xq, sx, w13q, s13, w2q, s2):
        I = w13q.shape[0] // 2
        return O.expert_forward(xq, sx, np.concatenate([w13q[I:], w13q[:I]]), np.concatenate([s13[s13.shape[0] // 2:], s13[:s13.shape[0] // 2]]), w2q, s2)
    assert _fails(pin_expert_hand_example, fwd_swapped)

    # quantisation without the 1e-4 floor
    def quant_nofloor(v):
        v = np.asarray(v, np.float32)
        b = v.reshape(v.shape[0], -1, 128)
        amax = np.abs(b).max(axis=2).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.float32(448.0) / amax
            sc = np.nan_to_num(b * r[..., None]).astype(np.float32)
        return O.e4m3_encode(sc).reshape(v.shape), (amax / np.float32(448.0)).astype(np.float32)
    assert _fails(pin_quant_special_cases, quant_nofloor)

    # rounding half away from zero instead of to even
    def enc_away(v):
        v = np.asarray(v, np.float32)
        out = O.e4m3_encode(v)
        a = np.abs(v).astype(np.float64)
        nxt = np.minimum((out & 0x7F).astype(np.int64) + 1, 0x7E)
        lo = O.e4m3_decode((out & 0x7F)); hi = O.e4m3_decode(nxt.astype(np.uint8))
        tie = (a == (lo + hi) / 2) & (a < 448)
        out = np.where(tie, nxt | (out & 0x80), out).astype(np.uint8)
        return out
    assert _fails(pin_encode_nearest_even, enc_away)

    # slots handed out in descending route id
    def route_desc(idx, E, R):
        T, K = idx.shape
        rr = O.route(idx[::-1, ::-1].copy(), E, R)
        return O.RouteResult(rr.counts, rr.src_map[::-1, ::-1].copy(), rr.routed, rr.dropped, rr.bad_id)
    assert _fails(pin_route_canonical, route_desc)

    # router weight dropped from combine
    def comb_noweight(out, src, w):
        return O.combine_fp64(out, src, np.ones_like(w))
    assert _fails(pin_combine_traced, comb_noweight)

    # per-source slots without the source's range offset (a packed prefix)
    def slots_noseg(idx, E, L, mt, src):
        res = O.route_source_slots(idx, E, L, mt, src)
        rr = O.route(idx, E, (E // L) * mt)
        return O.SourceSlotResult(res.counts, res.seg_counts, rr.src_map, res.dropped, res.bad_id)
    assert _fails(pin_source_slots_traced, slots_noseg)

    # slot range chosen by the destination rank instead of the source rank
    def slots_dest(idx, E, L, mt, src):
        return O.route_source_slots(idx, E, L, mt, np.asarray(idx)[:, 0] // L)
    assert _fails(pin_source_slots_traced, slots_dest)

    # combine with a fused multiply-add per term (one rounding per term)
    def comb_fma(out, src, w):
        T, K = src.shape
        acc = np.zeros((T, out.shape[1]), np.float64)
        for k in range(K):
            m = src[:, k] >= 0
            prod = w[m, k].astype(np.float64)[:, None] * out[src[m, k]].astype(np.float64)
            acc[m] = (acc[m].astype(np.float32).astype(np.float64) + prod).astype(np.float32)
        return O.f32_to_bf16_rne(acc.astype(np.float32))
    assert _fails(pin_combine_rounding, comb_fma)

    # combine accumulated in fp64 and rounded once
    def comb_wide(out, src, w):
        return O.f32_to_bf16_rne(O.combine_fp64(out, src, w).astype(np.float32))
    assert _fails(pin_combine_rounding, comb_wide)


def test_packed_offsets_page_example():
    """"SGLang Expert Compute Backend", §2.6: with compact storage expert 1's
    first row follows expert 0's 70th valid row; 82 valid rows in place of the
    256 capacity rows of the [70, 12] example."""
    off = O.packed_row_offsets([70, 12])
    assert off.tolist() == [0, 70, 82]
    assert off[-1] == 82 and 2 * 128 == 256


def test_packed_src_map_is_order_preserving_bijection():
    """Brute force over random routings: the packed map sends the kept routes
    of expert e, in slot order, onto consecutive rows starting at the sum of
    the earlier experts' counts, and covers [0, sum(counts)) exactly once."""
    rng = np.random.default_rng(11)
    for _ in range(30):
        E, R, T, K = int(rng.integers(1, 9)), int(rng.integers(1, 12)), int(rng.integers(0, 40)), 2
        K = min(K, E)
        idx = np.stack([rng.choice(np.arange(-1, E), size=K, replace=False) for _ in range(T)]) \
            if T else np.zeros((0, K), np.int64)
        r = O.route(idx, E, R)
        p = O.packed_src_map(r.src_map, r.counts, R)
        kept = p[p >= 0]
        assert sorted(kept.tolist()) == list(range(int(np.sum(r.counts))))
        start = 0
        for e in range(E):
            slots = sorted(int(q) - e * R for q in r.src_map.flatten() if q >= 0 and q // R == e)
            rows = sorted(int(pp) for q, pp in zip(r.src_map.flatten(), p.flatten()) if q >= 0 and q // R == e)
            assert rows == [start + s for s in slots]
            start += int(r.counts[e])


def test_interleaved_gateup_is_a_row_permutation():
    """With one scale for every weight block, interleaving the gate/up rows
    (row 2j gate j, row 2j+1 up j) must give exactly the standard expert: the
    same products and sums with G's columns permuted."""
    rng = np.random.default_rng(12)
    m, H, I = 5, 256, 256
    def codes(*shape):   # signed e4m3 codes of both signs, NaN codes (0x7F, 0xFF) excluded
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        c[(c & 0x7F) == 0x7F] = 0
        return c
    xq, w13, w2 = codes(m, H), codes(2 * I, H), codes(H, I)
    sx = rng.uniform(0.5, 2.0, size=(m, H // 128)).astype(np.float32) * 1e-3
    s13 = np.full((2 * I // 128, H // 128), 1e-3, np.float32)
    s2 = np.full((H // 128, I // 128), 2e-3, np.float32)
    inter = np.empty_like(w13)
    inter[0::2], inter[1::2] = w13[:I], w13[I:]
    out_std, zq_std, sz_std, _ = O.expert_forward(xq, sx, w13, s13, w2, s2)
    out_int, zq_int, sz_int, _ = O.expert_forward(xq, sx, inter, s13, w2, s2, interleaved=True)
    assert np.array_equal(zq_std, zq_int) and np.array_equal(sz_std, sz_int)
    assert np.array_equal(out_std, out_int)
    # reading the halves the other way round (up first) is not the same expert
    swapped = np.empty_like(w13)
    swapped[0::2], swapped[1::2] = w13[I:], w13[:I]
    out_bad, _, _, _ = O.expert_forward(xq, sx, swapped, s13, w2, s2, interleaved=True)
    assert not np.array_equal(out_bad, out_std)
