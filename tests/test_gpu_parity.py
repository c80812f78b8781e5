"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: dispatch (counts, src_map, the payload rows), the FP8 quantisation
bytes and scales, and combine (against the fp32 restatement).  Within 2e-2
max relative error per row (vs the fp64 oracle on the same quantised
operands): the grouped GEMMs and the whole layer.
"""
import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_grouped_topk_gb300 import api
from token_dispatch_grouped_topk_gb300 import workloads as W

from helpers import REL_TOL, assert_rows_close, f32, host_weights, oracle_expert_rows, u8

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api._lib.load()
    yield
    torch.cuda.synchronize()


def check_routing(idx, E, R, counts, src_map, status):
    """Counts, source map and status bit-exact against the oracle's
    canonical routing."""
    rr = O.route(idx.cpu().numpy(), E, R)
    assert counts.cpu().numpy().tolist() == rr.counts.tolist()
    assert np.array_equal(src_map.cpu().numpy(), rr.src_map)
    st = status.cpu().numpy()
    assert int(st[1]) == rr.dropped
    assert bool(st[0] & api.DEV_CAPACITY_DROPPED) == (rr.dropped > 0)
    assert bool(st[0] & api.DEV_BAD_EXPERT_ID) == rr.bad_id
    return rr


def check_dispatch(x, idx, E, R, recv, counts, src_map, status):
    """Bit-exact dispatch check against the oracle's canonical routing."""
    rr = check_routing(idx, E, R, counts, src_map, status)
    # payload: every kept route's row equals its token row, bit for bit
    sm = torch.from_numpy(rr.src_map).to(x.device).long()
    tok = torch.arange(x.shape[0], device=x.device)[:, None].expand_as(sm)
    keep = sm >= 0
    rows = recv.view(-1, x.shape[1])[sm[keep]]
    assert torch.equal(rows.view(torch.int16), x[tok[keep]].view(torch.int16))
    return rr


def check_dispatch_fp8(x, idx, E, R, xq, xs, counts, src_map, status, max_tokens=1024, seed=0):
    """The fused dispatch+quant path's outputs: routing bit-exact against the
    oracle; every kept route's e4m3 row and scales equal those of the other
    routes of its token (all K copies identical); and, on all tokens or a
    sample of max_tokens, the oracle's quantisation of the token row."""
    rr = check_routing(idx, E, R, counts, src_map, status)
    H = x.shape[1]
    q_rows, s_rows = xq.reshape(-1, H), xs.reshape(-1, H // 128)
    sm = torch.from_numpy(rr.src_map).to(x.device).long()
    keep = sm >= 0
    first = torch.where(keep, sm, torch.iinfo(torch.int64).max).min(dim=1).values
    tok = torch.arange(x.shape[0], device=x.device)[:, None].expand_as(sm)
    assert torch.equal(q_rows[sm[keep]], q_rows[first[tok[keep]]])
    assert torch.equal(s_rows[sm[keep]], s_rows[first[tok[keep]]])
    has = np.nonzero(keep.any(dim=1).cpu().numpy())[0]
    if len(has) > max_tokens:
        has = np.sort(np.random.default_rng(seed).choice(has, max_tokens, replace=False))
    codes, scales = O.quantize_rows(f32(x[torch.from_numpy(has).to(x.device)]))
    rows = first[torch.from_numpy(has).to(x.device)]
    assert np.array_equal(q_rows[rows].cpu().numpy(), codes)
    assert np.array_equal(s_rows[rows].cpu().numpy(), scales)
    return rr


# ---------------------------------------------------------------- dispatch

def test_dispatch_traced_scenario():
    d = W.make_layer_inputs("traced", seed=0, device=DEV, weights=False)
    wl = d["wl"]
    recv, counts, src_map, st = api.moe_dispatch(d["x"], d["topk_idx"], d["topk_w"], wl.E, wl.R)
    torch.cuda.synchronize()
    rr = check_dispatch(d["x"], d["topk_idx"], wl.E, wl.R, recv, counts, src_map, st)
    assert counts.cpu().tolist() == [111, 1, 0, 0, 0, 0, 1, 111]
    assert src_map[21].cpu().tolist() == [1 * 128, 6 * 128]
    assert rr.dropped == 0


@pytest.mark.parametrize("E,K", [(1, 1), (3, 2), (8, 2), (8, 8), (33, 5), (256, 8), (64, 32)])
def test_dispatch_random_small(E, K):
    g = torch.Generator().manual_seed(E * 100 + K)
    for T in (0, 1, 17, 300):
        for R in (1, 5, 64):
            H = 128 if T > 100 else 256
            idx = torch.randint(-1, E, (T, K), generator=g)
            if T > 3:
                idx[3, 0] = E + 4  # invalid id: reported, route ignored
            x = torch.randn(T, H, generator=g).to(torch.bfloat16)
            xd, idd = x.to(DEV), idx.to(DEV)
            recv, counts, src_map, st = api.moe_dispatch(xd, idd, None, E, R)
            torch.cuda.synchronize()
            check_dispatch(xd, idd, E, R, recv, counts, src_map, st)


@pytest.mark.parametrize("T,K", [(512, 8), (513, 8), (4096, 1), (4097, 1)])
def test_dispatch_single_pass_threshold(T, K):
    """Both sides of the single-kernel threshold (T*K <= 4096 routes: every
    block counts the routes before its own; above it: histogram, scan,
    scatter) give the oracle's canonical slots, counts and status, with
    capacity drops and an invalid id, padded and packed, int64 and int32 ids."""
    E, R, H = 40, 60, 256
    g = torch.Generator().manual_seed(T * 7 + K)
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[:, 0] = torch.randint(0, 4, (T,), generator=g)
    idx[T // 2, 0] = E + 1
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    xd, idd = x.to(DEV), idx.to(DEV)
    recv, counts, src_map, st = api.moe_dispatch(xd, idd, None, E, R)
    torch.cuda.synchronize()
    rr = check_dispatch(xd, idd, E, R, recv, counts, src_map, st)
    assert rr.dropped > 0 and rr.bad_id
    precv, pc, pm, pst = api.moe_dispatch_packed(xd, idd.to(torch.int32), None, E, R)
    torch.cuda.synchronize()
    assert torch.equal(pc, counts) and torch.equal(pst, st)
    assert np.array_equal(pm.cpu().numpy(), O.packed_src_map(rr.src_map, rr.counts, R))


def test_dispatch_empty_rank_resets_counts():
    counts = torch.full((8,), 99, dtype=torch.int32, device=DEV)
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(0, 2, dtype=torch.int64, device=DEV)
    _, counts, src_map, st = api.moe_dispatch(x, idx, None, 8, 128, counts=counts)
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == [0] * 8 and st.cpu().tolist() == [0, 0]
    assert src_map.shape == (0, 2)


# ------------------------------------------------------------------- quant

def test_quantize_bit_exact_ragged():
    g = torch.Generator().manual_seed(5)
    E, R, H = 5, 200, 640
    counts = torch.tensor([200, 0, 1, 77, 129], dtype=torch.int32)
    recv = (torch.randn(E, R, H, generator=g) * torch.rand(E, R, 1, generator=g) * 30).to(torch.bfloat16)
    recv[2, 0, :128] = 0.0                   # floor case
    recv[3, 5, 128:256] = 2.5                # constant group
    recv[3, 6, 256:384] = 1e-30              # tiny values below the floor
    for e in range(E):
        recv[e, counts[e]:] = float("nan")   # capacity rows must never be read
    rd, cd = recv.to(DEV), counts.to(DEV)
    xq0 = torch.full((E, R, H), 0xAB, dtype=torch.uint8, device=DEV)
    xq, xs = api.moe_quantize_fp8(rd, cd, xq=xq0)
    torch.cuda.synchronize()
    xq_h, xs_h = u8(xq), f32(xs)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            assert np.all(xq_h[e] == 0xAB)
            continue
        codes, scales = O.quantize_rows(f32(recv[e, :c]))
        assert np.array_equal(xq_h[e, :c], codes)
        assert np.array_equal(xs_h[e, :c], scales)
        assert np.all(xq_h[e, c:] == 0xAB)   # capacity rows untouched


# ------------------------------------------------- fused dispatch + quant

@pytest.mark.parametrize("T,E,K,R,H", [(300, 33, 5, 40, 640), (4, 8, 2, 4, 256), (2000, 64, 8, 200, 1024),
                                       (3000, 16, 2, 500, 256), (2100, 12, 1, 300, 1024),
                                       (5000, 12, 1, 500, 1024)])
def test_dispatch_quant_matches_dispatch_then_quant(T, E, K, R, H):
    """moe_dispatch_quant writes exactly the bytes moe_quantize_fp8 writes on
    moe_dispatch's receive rows (and the oracle's quantisation of the token
    rows), with the same counts, source map and status.  The shapes take every
    form of the kernel on a 152-SM GB300: single pass with 16 and no preloaded
    loads per lane (first two, fifth), three launches with 8, 16 and none
    (third, fourth, sixth)."""
    g = torch.Generator().manual_seed(T + E)
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[:, 0] = torch.randint(0, 3, (T,), generator=g)     # hot experts: capacity drops
    idx[1, K - 1] = E + 9                                   # invalid id
    x = (torch.randn(T, H, generator=g) * torch.rand(T, 1, generator=g) * 5).to(torch.bfloat16)
    x[2, :128] = 0.0
    xd, idd = x.to(DEV), idx.to(DEV)
    recv, c1, m1, s1 = api.moe_dispatch(xd, idd, None, E, R)
    xq1, xs1 = api.moe_quantize_fp8(recv, c1)
    xq2, xs2, c2, m2, s2 = api.moe_dispatch_quant(xd, idd, None, E, R)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(m1, m2) and torch.equal(s1, s2)
    rr = O.route(idx.numpy(), E, R)
    assert np.array_equal(m2.cpu().numpy(), rr.src_map)
    rows = torch.from_numpy(rr.src_map[rr.src_map >= 0]).long()
    tok = torch.from_numpy(np.nonzero(rr.src_map >= 0)[0]).long()
    got_q = xq2.view(-1, H).cpu()[rows]
    got_s = xs2.view(-1, H // 128).cpu()[rows]
    assert torch.equal(got_q, xq1.view(-1, H).cpu()[rows])
    assert torch.equal(got_s, xs1.view(-1, H // 128).cpu()[rows])
    codes, scales = O.quantize_rows(f32(x)[tok.numpy()])
    assert np.array_equal(got_q.numpy(), codes) and np.array_equal(got_s.numpy(), scales)


@pytest.mark.parametrize("name", ["traced", "decode"])
def test_layer_fused_path_bit_identical(name):
    d = W.make_layer_inputs(name, seed=5, device=DEV)
    wl = d["wl"]
    args = (d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    y1 = buf.forward(*args, fused=False).clone()
    y2 = buf.forward(*args)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert buf.dev_status.cpu().tolist()[0] & api.DEV_TIMEOUT == 0


# ------------------------------------------------------------------- GEMMs

def _expert_setup(E, R, H, I, counts, seed):
    g = torch.Generator().manual_seed(seed)
    recv = torch.randn(E, R, H, generator=g).to(torch.bfloat16)
    for e in range(E):
        recv[e, counts[e]:] = float("nan")
    w13, s13, w2, s2 = W.expert_weights(E, H, I, seed, "cpu")
    return recv, w13, s13, w2, s2


def _check_expert_compute(E, R, H, I, counts, seed):
    recv, w13, s13, w2, s2 = _expert_setup(E, R, H, I, counts, seed)
    cd = torch.tensor(counts, dtype=torch.int32, device=DEV)
    rd = recv.to(DEV)
    sentinel = torch.full((E, R, H), 3.0, dtype=torch.bfloat16, device=DEV)
    # step by step through the stage entry points
    xq, xs = api.moe_quantize_fp8(rd, cd)
    zq, zs = api.moe_gemm_gateup_silu(xq, xs, cd, w13.to(DEV), s13.to(DEV))
    out = api.moe_gemm_down(zq, zs, cd, w2.to(DEV), s2.to(DEV), out=sentinel.clone())
    # and the fused call
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    out2 = api.moe_expert_compute(rd, cd, w13.to(DEV), s13.to(DEV), w2.to(DEV), s2.to(DEV),
                                  out=sentinel.clone(), dev_status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0]
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    zq_h, zs_h, out_h = u8(zq), f32(zs), f32(out)
    worst = 0.0
    for e in range(E):
        c = counts[e]
        assert np.all(out_h[e, c:] == 3.0), "capacity rows of out were written"
        if c == 0:
            continue
        xqo, sxo = O.quantize_rows(f32(recv[e, :c]))
        ref, zq_ref, sz_ref, _ = O.expert_forward(xqo, sxo, u8(w13[e]), f32(s13[e]), u8(w2[e]), f32(s2[e]))
        # Z: scales agree to fp32 rounding noise, codes to within one e4m3 step
        assert np.allclose(zs_h[e, :c], sz_ref, rtol=1e-4, atol=0)
        dz = np.abs(O.e4m3_decode(zq_h[e, :c]) - O.e4m3_decode(zq_ref))
        step = np.maximum(np.abs(O.e4m3_decode(zq_ref)), 2.0 ** -6) * 2.0 ** -3
        assert np.all(dz <= step + 1e-12)
        assert np.mean(zq_h[e, :c] != zq_ref) < 0.01
        worst = max(worst, assert_rows_close(out_h[e, :c], ref, what=f"expert {e}"))
    return worst


def test_gemm_unit_example():
    """The pages' [70, 12] example: 2 experts, R=128, H=256, I=128; capacity
    rows are NaN and must not leak."""
    _check_expert_compute(2, 128, 256, 128, [70, 12], seed=3)


def test_expert_compute_multi_tile_ragged():
    _check_expert_compute(4, 384, 512, 384, [300, 129, 0, 17], seed=4)


def test_expert_compute_bn128_tail():
    """H = 384 is not a multiple of 256: the down GEMM uses 128-wide tiles."""
    _check_expert_compute(3, 256, 384, 256, [256, 1, 130], seed=5)


def test_expert_compute_capacity_not_multiple_of_tile():
    _check_expert_compute(3, 200, 256, 128, [200, 199, 64], seed=6)


@pytest.mark.parametrize("H", [512, 384])
def test_expert_compute_activation_box_boundaries(H):
    """Blocks of 1..32, 33..64 and 65..128 valid rows fetch 32-, 64- and
    128-row activation boxes: both sides of each boundary, alone and after
    full blocks, with 256-wide (H=512) and 128-wide (H=384) down tiles."""
    counts = [1, 31, 32, 33, 63, 64, 65, 127, 129, 192, 193, 256, 0]
    _check_expert_compute(len(counts), 256, H, 256, counts, seed=11)


@pytest.mark.parametrize("H", [512, 384])
def test_expert_compute_short_blocks_only(H):
    """No expert above 64 rows: every tile fetches a short activation box,
    several tiles per CTA, with K groups rotating through both accumulator
    buffers."""
    counts = [1, 64, 33, 0, 17, 64, 2, 40, 63, 5, 64, 31]
    _check_expert_compute(len(counts), 64, H, 512, counts, seed=12)


@pytest.mark.parametrize("E,R,H,I,seed", [(5, 384, 512, 256, 21), (48, 256, 1024, 512, 22),
                                          (3, 256, 384, 256, 23), (1, 1024, 256, 1024, 24),
                                          (200, 128, 256, 128, 25)])
def test_gemm_gateup_down_matches_stage_calls(E, R, H, I, seed):
    """Both GEMMs in one launch (down tiles of a block start once that block's
    gate/up tiles are done) against the two stage launches: Z codes, Z scales
    and out bit-identical on the valid rows, capacity rows of out untouched;
    three launches in a row reuse one scratch (each resets it); the packed
    layout on the same rows gives the same rows.  H = 384 takes the two-launch
    form (128-wide down tiles).  E = 200 with H = 256, I = 128 makes tiles of one
    or two K groups: the producer runs far ahead through the tile ring and many
    down tiles reach their block's wait."""
    g = torch.Generator().manual_seed(seed)
    counts = torch.randint(0, R + 1, (E,), generator=g)
    counts[0] = R
    if E > 2:
        counts[1] = 0
    recv, w13, s13, w2, s2 = _expert_setup(E, R, H, I, counts.tolist(), seed)
    cd = counts.to(torch.int32).to(DEV)
    w13, s13, w2, s2 = (t.to(DEV) for t in (w13, s13, w2, s2))
    xq, xs = api.moe_quantize_fp8(recv.to(DEV), cd)
    zq1, zs1 = api.moe_gemm_gateup_silu(xq, xs, cd, w13, s13)
    out1 = api.moe_gemm_down(zq1, zs1, cd, w2, s2)
    sentinel = torch.full((E, R, H), 3.0, dtype=torch.bfloat16, device=DEV)
    zq2 = torch.zeros_like(zq1)
    zs2 = torch.zeros_like(zs1)
    sync = torch.empty(max(256, api._lib.load().moe_gemm_gateup_down_sync_size(E, R, 0)),
                       dtype=torch.uint8, device=DEV)
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    outs = []
    for _ in range(3):
        outs.append(api.moe_gemm_gateup_down(xq, xs, cd, w13, s13, w2, s2, zq=zq2, zs=zs2,
                                             out=sentinel.clone(), sync=sync, dev_status=st,
                                             gemm_launch="one"))
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0]
    valid = torch.arange(R).unsqueeze(0) < counts.unsqueeze(1)          # [E, R]
    vd = valid.to(DEV)
    assert torch.equal(zq1[vd], zq2[vd]) and torch.equal(zs1[vd], zs2[vd])
    for out2 in outs:
        assert torch.equal(out1[vd].view(torch.int16), out2[vd].view(torch.int16))
        assert bool((out2[~vd] == 3.0).all()), "capacity rows of out were written"
    # packed layout: the valid rows back to back
    xq_p, xs_p = xq[vd].contiguous(), xs[vd].contiguous()
    rows = xq_p.shape[0]
    if rows > 0:
        for form in ("one", "two"):
            out_p = api.moe_gemm_gateup_down(xq_p, xs_p, cd, w13, s13, w2, s2, R=R, dev_status=st,
                                             gemm_launch=form)
            torch.cuda.synchronize()
            assert st.cpu().tolist() == [0, 0]
            assert torch.equal(out_p.view(torch.int16), out1[vd].view(torch.int16)), form


def test_gemm_gateup_down_two_streams_at_once():
    """Two one-launch GEMMs on two streams at the same time, so their
    persistent CTAs compete for the SMs.  Tiles are taken in list order only by
    CTAs that are running, so a down tile never waits on a gate/up tile held by
    a CTA that has not started.  Both finish without a timeout and equal their
    results run alone."""
    E, R, H, I = 24, 512, 1024, 512
    dev = torch.device(DEV)
    runs = []
    for seed in (31, 32):
        g = torch.Generator().manual_seed(seed)
        counts = torch.randint(0, R + 1, (E,), generator=g)
        recv, w13, s13, w2, s2 = _expert_setup(E, R, H, I, counts.tolist(), seed)
        cd = counts.to(torch.int32).to(DEV)
        w13, s13, w2, s2 = (t.to(DEV) for t in (w13, s13, w2, s2))
        xq, xs = api.moe_quantize_fp8(recv.to(DEV), cd)
        alone = api.moe_gemm_gateup_down(xq, xs, cd, w13, s13, w2, s2, gemm_launch="one")
        runs.append(dict(args=(xq, xs, cd, w13, s13, w2, s2), alone=alone, cd=counts))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=dev) for _ in runs]
    st = [torch.zeros(2, dtype=torch.int32, device=DEV) for _ in runs]
    outs = [None, None]
    for rep in range(3):
        for i, (r, s) in enumerate(zip(runs, streams)):
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                outs[i] = api.moe_gemm_gateup_down(*r["args"], dev_status=st[i], stream=s,
                                                   gemm_launch="one")
        torch.cuda.synchronize()
        for i, r in enumerate(runs):
            assert st[i].cpu().tolist() == [0, 0]
            vd = (torch.arange(R).unsqueeze(0) < r["cd"].unsqueeze(1)).to(DEV)
            assert torch.equal(outs[i][vd].view(torch.int16), r["alone"][vd].view(torch.int16))


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_layer_gemm_launch_forms_bit_identical(name):
    """The layer with its GEMMs forced into one launch and into two launches
    gives the same bytes (the default picks one of the two by tile count)."""
    d = W.make_layer_inputs(name, seed=9, device=DEV)
    wl = d["wl"]
    args = (d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    ys = []
    for form in ("one", "two", None):
        buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV),
                                  gemm_launch=form)
        ys.append(buf.forward(*args).clone())
        torch.cuda.synchronize()
        assert buf.dev_status[0].item() & api.DEV_TIMEOUT == 0
        del buf
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    assert torch.equal(ys[0].view(torch.int16), ys[2].view(torch.int16))


# ------------------------------------------------------------------ combine

def test_combine_bit_exact():
    g = torch.Generator().manual_seed(7)
    E, R, H, T, K = 6, 50, 384, 77, 4
    out = (torch.randn(E, R, H, generator=g) * 3).to(torch.bfloat16)
    src = torch.randint(-1, E * R, (T, K), generator=g).to(torch.int32)
    src[5] = -1                               # token with no kept route
    w = torch.rand(T, K, generator=g)
    y = api.moe_combine(out.to(DEV), src.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    want = O.combine_f32_sequential(f32(out).reshape(E * R, H), src.numpy(), w.numpy())
    assert np.array_equal(f32(y), want)
    assert np.all(f32(y)[5] == 0)


def test_identity_experts_return_input():
    d = W.make_layer_inputs("traced", seed=1, device=DEV, weights=False)
    wl = d["wl"]
    recv, counts, src_map, _ = api.moe_dispatch(d["x"], d["topk_idx"], d["topk_w"], wl.E, wl.R)
    y = api.moe_combine(recv, src_map, d["topk_w"])   # out := recv
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), d["x"].view(torch.int16))


# -------------------------------------------------------------- whole layer

def _layer_oracle(d, tokens=None):
    wl = d["wl"]
    x = f32(d["x"])
    idx = d["topk_idx"].cpu().numpy()
    w = d["topk_w"].cpu().numpy()
    rr = O.route(idx, wl.E, wl.R)
    toks = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    experts = sorted({int(idx[t, k]) for t in toks for k in range(wl.K) if rr.src_map[t, k] >= 0})
    wts = host_weights(d, experts)
    y = np.zeros((len(toks), wl.H))
    route_out = {}
    for e in experts:
        sel = [(i, k) for i, t in enumerate(toks) for k in range(wl.K)
               if idx[t, k] == e and rr.src_map[t, k] >= 0]
        rows = oracle_expert_rows(x[[toks[i] for i, _ in sel]], wts[e])
        for (i, k), r in zip(sel, rows):
            y[i] += float(w[toks[i], k]) * r
            route_out[(int(toks[i]), k)] = r
    return y, rr, route_out


def test_layer_traced_scenario():
    d = W.make_layer_inputs("traced", seed=0, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    y = buf.forward(d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    torch.cuda.synchronize()
    y_ref, rr, _ = _layer_oracle(d)
    assert_rows_close(f32(y), y_ref, what="y")
    # token 21 = 0.25 * F1(x) + 0.75 * F6(x)
    assert buf.counts.cpu().tolist() == [111, 1, 0, 0, 0, 0, 1, 111]


def test_graph_replay_changes_routes():
    """Replay of one captured graph reads the routes current at replay: switching
    token 21 from [E1, E6] to [E0, E7] moves counts 111/1/1/111 -> 112/0/0/112
    and the output follows (the pages' replay example)."""
    d = W.make_layer_inputs("traced", seed=0, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    x, idx, w = d["x"].clone(), d["topk_idx"].clone(), d["topk_w"].clone()
    args = (d["w13"], d["s13"], d["w2"], d["s2"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        buf.forward(x, idx, w, *args)         # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        buf.forward(x, idx, w, *args)
    swapped, _ = W.traced_routes(0, swap_token_21=True)
    idx.copy_(swapped.to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    assert [int(buf.counts[e]) for e in (0, 1, 6, 7)] == [112, 0, 0, 112]
    d2 = dict(d, topk_idx=idx)
    y_ref, _, _ = _layer_oracle(d2)
    assert_rows_close(f32(buf.y), y_ref, what="replayed y")
    idx.copy_(d["topk_idx"])
    graph.replay()
    torch.cuda.synchronize()
    assert [int(buf.counts[e]) for e in (0, 1, 6, 7)] == [111, 1, 1, 111]


def test_layer_decode_config():
    """Decode-shaped layer, full size (T=256, E=64, top-8, H=4096, I=1536,
    R=256), both layer paths: dispatch (BF16 rows, or FP8 rows and scales on
    the fused path) bit-exact, y the same bytes, every fourth token's output
    against the oracle."""
    d = W.make_layer_inputs("decode", seed=0, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    args = (d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    y_sep = buf.forward(*args, fused=False).clone()
    torch.cuda.synchronize()
    check_dispatch(d["x"], d["topk_idx"], wl.E, wl.R, buf.recv, buf.counts, buf.src_map, buf.dev_status)
    y = buf.forward(*args)
    torch.cuda.synchronize()
    xq, xs, _, _ = buf.workspace_views()
    check_dispatch_fp8(d["x"], d["topk_idx"], wl.E, wl.R, xq, xs, buf.counts, buf.src_map, buf.dev_status)
    assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16))
    toks = np.arange(0, wl.T, 4)
    y_ref, _, _ = _layer_oracle(d, toks)
    assert_rows_close(f32(y)[toks], y_ref, what="decode y")


@pytest.mark.parametrize("graph,layout", [(False, "padded"), (True, "padded"),
                                          (True, "source_slots")])
def test_host_pipeline_matches_forward(graph, layout):
    """api.HostPipeline (pinned host in/out, copies of neighbouring steps
    overlapped with compute, two device slots; eager, or each slot's layer
    captured once in a CUDA graph and replayed) returns, for every step, the
    bytes a plain forward on device inputs returns; five steps reuse each slot
    at least twice, with a different routing per step.  The per-source lane
    forms its FP8 slots in the pipeline's first (eager) step, before the
    capture."""
    d = W.make_layer_inputs("decode", seed=0, device=DEV)
    wl = d["wl"]
    dev = torch.device(DEV)

    def lane():
        if layout == "padded":
            return api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
        mt = wl.T // wl.W
        return api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.W * mt, dev, source_slots=mt,
                                   L=wl.L)
    buf = lane()
    steps = []
    for i in range(5):
        idx, w = W.router(wl.T, wl.E, wl.K, W.router_bias(wl, 10 + i, "cpu"), 20 + i, "cpu")
        x = W.activations(wl.T, wl.H, 30 + i, "cpu")
        steps.append((x, idx, w))
    want = []
    for x, idx, w in steps:
        y = buf.forward(x.to(dev), idx.to(dev), w.to(dev), d["w13"], d["s13"], d["w2"], d["s2"])
        want.append(y.cpu())
    buf = lane()
    pipe = api.HostPipeline(buf, graph=graph)
    outs = [torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory() for _ in steps]
    pinned = [(x.pin_memory(), idx.pin_memory(), w.pin_memory()) for x, idx, w in steps]
    for (x, idx, w), y_h in zip(pinned, outs):
        pipe.submit(x, idx, w, y_h, d["w13"], d["s13"], d["w2"], d["s2"])
    pipe.synchronize()
    for i, (got, ref) in enumerate(zip(outs, want)):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"step {i}"
    with pytest.raises(ValueError):
        pipe.submit(steps[0][0], *pinned[0][1:], outs[0], d["w13"], d["s13"], d["w2"], d["s2"])


def _sampled_out_check(d, buf, n_routes, seed):
    """Expert outputs of sampled kept routes, one by one against the oracle."""
    wl = d["wl"]
    rng = np.random.default_rng(seed)
    src = buf.src_map.cpu().numpy()
    idx = d["topk_idx"].cpu().numpy()
    kept = np.argwhere(src >= 0)
    pick = kept[rng.choice(len(kept), size=min(n_routes, len(kept)), replace=False)]
    experts = sorted({int(idx[t, k]) for t, k in pick})
    wts = host_weights(d, experts)
    x = d["x"]
    out_flat = buf.out.view(-1, wl.H)
    for e in experts:
        sel = [(t, k) for t, k in pick if idx[t, k] == e]
        rows = oracle_expert_rows(f32(x[[t for t, _ in sel]]), wts[e])
        got = f32(out_flat[[int(src[t, k]) for t, k in sel]])
        assert_rows_close(got, rows, what=f"expert {e} sampled rows")


def test_layer_prefill_config_and_split():
    """Prefill-shaped Zipf-skewed layer (T=4096, E=128, R=2048): dispatch
    bit-exact (with capacity drops), sampled expert rows against the oracle,
    combine against the fp32 restatement, and the two-micro-batch split: rows
    of tokens whose routes are kept in both runs are bit-identical."""
    d = W.make_layer_inputs("prefill", seed=0, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    args = (d["w13"], d["s13"], d["w2"], d["s2"])
    y = buf.forward(d["x"], d["topk_idx"], d["topk_w"], *args).clone()
    torch.cuda.synchronize()
    xq, xs, _, _ = buf.workspace_views()
    rr = check_dispatch_fp8(d["x"], d["topk_idx"], wl.E, wl.R, xq, xs, buf.counts, buf.src_map,
                            buf.dev_status, max_tokens=wl.T)
    assert rr.dropped > 0
    y_sep = buf.forward(d["x"], d["topk_idx"], d["topk_w"], *args, fused=False).clone()
    torch.cuda.synchronize()
    check_dispatch(d["x"], d["topk_idx"], wl.E, wl.R, buf.recv, buf.counts, buf.src_map, buf.dev_status)
    assert torch.equal(y_sep.view(torch.int16), y.view(torch.int16))
    _sampled_out_check(d, buf, 48, seed=1)
    want = O.combine_f32_sequential(f32(buf.out).reshape(-1, wl.H), buf.src_map.cpu().numpy(),
                                    d["topk_w"].cpu().numpy())
    assert np.array_equal(f32(y), want)
    # split into two lanes of 2048 tokens
    half = wl.T // 2
    lanes = [api.MoeLayerBuffers(half, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV)) for _ in range(2)]
    ys = [lanes[i].forward(d["x"][i * half:(i + 1) * half], d["topk_idx"][i * half:(i + 1) * half],
                           d["topk_w"][i * half:(i + 1) * half], *args) for i in range(2)]
    torch.cuda.synchronize()
    y_split = torch.cat(ys)
    full_kept = (buf.src_map >= 0) | (d["topk_idx"] < 0)
    split_map = torch.cat([lane.src_map for lane in lanes])
    split_kept = (split_map >= 0) | (d["topk_idx"] < 0)
    same = (full_kept.all(1) & split_kept.all(1))
    assert int(same.sum()) > wl.T // 4
    assert torch.equal(y_split[same].view(torch.int16), y[same].view(torch.int16))


@pytest.mark.parametrize("fused", [True, False])
def test_two_batch_overlap_equals_serial_split(fused):
    """The overlapped two-micro-batch schedule (two lanes, two streams) writes
    exactly what the serial split writes, and equals the unsplit layer on every
    token whose routes are kept in both; with the fused dispatch+quant stages
    and with the separate ones."""
    d = W.make_layer_inputs("prefill", seed=4, device=DEV)
    wl = d["wl"]
    args = (d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    tbo = api.TwoBatchOverlap(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV), fused=fused)
    y_serial = tbo.forward(*args, overlap=False).clone()
    y_over = tbo.forward(*args, overlap=True).clone()
    full = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    y_full = full.forward(*args)
    torch.cuda.synchronize()
    assert torch.equal(y_serial.view(torch.int16), y_over.view(torch.int16))
    kept_full = ((full.src_map >= 0) | (d["topk_idx"] < 0)).all(1)
    split_map = torch.cat([lane.src_map for lane in tbo.lanes])
    kept_split = ((split_map >= 0) | (d["topk_idx"] < 0)).all(1)
    same = kept_full & kept_split
    assert torch.equal(y_over[same].view(torch.int16), y_full[same].view(torch.int16))
    for lane in tbo.lanes:
        assert lane.dev_status[0].item() & api.DEV_TIMEOUT == 0


def test_two_batch_overlap_graph_replay():
    """The overlapped two-micro-batch schedule captured in one CUDA graph (the
    side streams fork from and join the capturing stream): replays equal the
    eager overlapped forward, also after new routes are copied into the
    captured input buffers."""
    d = W.make_layer_inputs("prefill", seed=6, device=DEV)
    d2 = W.make_layer_inputs("prefill", seed=7, device=DEV)
    wl = d["wl"]
    dev = torch.device(DEV)
    tbo = api.TwoBatchOverlap(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    x, idx, w = d["x"].clone(), d["topk_idx"].clone(), d["topk_w"].clone()
    wts = (d["w13"], d["s13"], d["w2"], d["s2"])
    tbo.forward(x, idx, w, *wts, overlap=True)          # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tbo.forward(x, idx, w, *wts, overlap=True)
    ref = api.TwoBatchOverlap(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    for inputs in (d, d2):
        x.copy_(inputs["x"])
        idx.copy_(inputs["topk_idx"])
        w.copy_(inputs["topk_w"])
        g.replay()
        got = tbo.y.clone()
        want = ref.forward(inputs["x"], inputs["topk_idx"], inputs["topk_w"], *wts, overlap=True)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        for lane in tbo.lanes:
            assert lane.dev_status[0].item() & api.DEV_TIMEOUT == 0


def test_layer_large_config_sampled():
    """Large layer (T=16384, E=256, H=7168, I=2048, R=4096, ~11 GB of FP8
    weights), in the launch configuration the benchmark times (the fused
    dispatch+quant path in a CUDA graph): routing bit-exact, the FP8 rows of
    512 sampled tokens against the oracle's quantisation (and every copy of a
    token's row identical), sampled expert rows against the oracle, combine
    bit-exact against the fp32 restatement, two graph replays with new
    routing."""
    d = W.make_layer_inputs("large", seed=0, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    args = (d["w13"], d["s13"], d["w2"], d["s2"])
    idx, w = d["topk_idx"].clone(), d["topk_w"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        buf.forward(d["x"], idx, w, *args)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        buf.forward(d["x"], idx, w, *args)
    for seed in (0, 11):
        i2, w2_ = W.router(wl.T, wl.E, wl.K, W.router_bias(wl, seed, DEV), seed + 1, DEV)
        idx.copy_(i2)
        w.copy_(w2_)
        graph.replay()
        torch.cuda.synchronize()
        xq, xs, _, _ = buf.workspace_views()
        check_dispatch_fp8(d["x"], idx, wl.E, wl.R, xq, xs, buf.counts, buf.src_map, buf.dev_status,
                           max_tokens=512, seed=seed)
        dd = dict(d, topk_idx=idx, topk_w=w)
        _sampled_out_check(dd, buf, 24, seed=seed)
        toks = np.random.default_rng(seed).choice(wl.T, 512, replace=False)
        sm = buf.src_map.cpu().numpy()[toks]
        uniq, inv = np.unique(sm[sm >= 0], return_inverse=True)
        compact = np.full_like(sm, -1)
        compact[sm >= 0] = inv
        rows = f32(buf.out.view(-1, wl.H)[torch.from_numpy(uniq).to(DEV).long()])
        want = O.combine_f32_sequential(rows, compact, w.cpu().numpy()[toks])
        assert np.array_equal(f32(buf.y)[toks], want)


@pytest.mark.parametrize("fused", [True, False])
def test_layer_degenerate_routings(fused):
    """Both layer paths on the degenerate inputs: no tokens (counts reset,
    nothing launched past the dispatch), every route a padding route (no
    expert rows, y = 0), and every route to one expert past its capacity
    (drops counted, kept rows against the oracle)."""
    E, K, H, I, R = 4, 2, 256, 128, 8
    dev = torch.device(DEV)
    w13, s13, w2, s2 = (t.to(DEV) for t in W.expert_weights(E, H, I, 17, "cpu"))
    # no tokens
    buf = api.MoeLayerBuffers(0, E, K, H, I, R, dev)
    buf.counts.fill_(99)
    y = buf.forward(torch.empty(0, H, dtype=torch.bfloat16, device=DEV),
                    torch.empty(0, K, dtype=torch.int64, device=DEV),
                    torch.empty(0, K, device=DEV), w13, s13, w2, s2, fused=fused)
    torch.cuda.synchronize()
    assert y.shape == (0, H)
    assert buf.counts.cpu().tolist() == [0] * E and buf.dev_status.cpu().tolist() == [0, 0]
    # every route a padding route
    T = 40
    g = torch.Generator().manual_seed(19)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.rand(T, K, generator=g).to(DEV)
    buf = api.MoeLayerBuffers(T, E, K, H, I, R, dev)
    buf.y.fill_(7.0)
    y = buf.forward(x, torch.full((T, K), -1, dtype=torch.int64, device=DEV), w, w13, s13, w2, s2,
                    fused=fused)
    torch.cuda.synchronize()
    assert buf.counts.cpu().tolist() == [0] * E and buf.dev_status.cpu().tolist() == [0, 0]
    assert bool((y.float() == 0).all())
    assert bool((buf.src_map == -1).all())
    # every route to expert 2: R of T*K kept, the rest dropped
    idx = torch.full((T, K), 2, dtype=torch.int64)
    idx[:, 1] = -1
    buf = api.MoeLayerBuffers(T, E, K, H, I, R, dev)
    y = buf.forward(x, idx.to(DEV), w, w13, s13, w2, s2, fused=fused)
    torch.cuda.synchronize()
    rr = O.route(idx.numpy(), E, R)
    assert buf.counts.cpu().tolist() == rr.counts.tolist() == [0, 0, R, 0]
    assert buf.dev_status.cpu().tolist() == [api.DEV_CAPACITY_DROPPED, T - R]
    assert np.array_equal(buf.src_map.cpu().numpy(), rr.src_map)
    kept = np.nonzero(rr.src_map[:, 0] >= 0)[0]
    wts = host_weights({"w13": w13, "s13": s13, "w2": w2, "s2": s2}, [2])
    ref = oracle_expert_rows(f32(x[torch.from_numpy(kept).to(DEV)]), wts[2])
    got = f32(buf.out.view(-1, H)[torch.from_numpy(rr.src_map[kept, 0]).long().to(DEV)])
    assert_rows_close(got, ref, what="one expert's kept rows")
    yk = f32(y)
    assert np.all(yk[np.setdiff1d(np.arange(T), kept)] == 0)


@pytest.mark.parametrize("T,E,K,H,I,R", [(50, 1, 1, 384, 128, 64), (90, 40, 32, 640, 256, 80),
                                         (33, 3, 2, 128, 384, 16), (64, 4, 2, 16384, 128, 48),
                                         (48, 4, 2, 128, 16384, 40)])
def test_layer_paths_odd_shapes(T, E, K, H, I, R):
    """The fused and separate layer paths on shapes off the benchmarked grid:
    one expert with top-1, top-32 of 40 experts, H % 256 = 128 (128-column
    down tiles), H = 128 (one K group), a single gate/up tile per block, and
    the largest hidden and intermediate sizes the library takes (16384, with
    the other side at one 128-group); y the same bytes on both paths and every
    kept route against the oracle."""
    dev = torch.device(DEV)
    g = torch.Generator().manual_seed(T + E + K)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)])
    idx[0, 0] = -1
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.rand(T, K, generator=g).to(DEV)
    w13, s13, w2, s2 = (t.to(DEV) for t in W.expert_weights(E, H, I, T, "cpu"))
    buf = api.MoeLayerBuffers(T, E, K, H, I, R, dev)
    y_sep = buf.forward(x, idx.to(DEV), w, w13, s13, w2, s2, fused=False).clone()
    y = buf.forward(x, idx.to(DEV), w, w13, s13, w2, s2)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16))
    rr = O.route(idx.numpy(), E, R)
    assert np.array_equal(buf.src_map.cpu().numpy(), rr.src_map)
    wts = host_weights({"w13": w13, "s13": s13, "w2": w2, "s2": s2}, range(E))
    src = rr.src_map
    for e in range(E):
        tk = np.argwhere((idx.numpy() == e) & (src >= 0))
        if len(tk) == 0:
            continue
        ref = oracle_expert_rows(f32(x[torch.from_numpy(tk[:, 0]).to(DEV)]), wts[e])
        got = f32(buf.out.view(-1, H)[torch.from_numpy(src[tk[:, 0], tk[:, 1]]).long().to(DEV)])
        assert_rows_close(got, ref, what=f"expert {e}")


def test_layer_max_experts():
    """The largest expert count the library takes (E = 1024: the per-expert
    tables in shared memory at their limit), top-8 over 400 tokens with an 8-row
    capacity (drops): routing bit-exact against the oracle, fused, separate and
    packed layer paths the same bytes, and the kept routes of every 16th expert
    against the oracle."""
    T, E, K, H, I, R = 400, 1024, 8, 256, 128, 8
    dev = torch.device(DEV)
    g = torch.Generator().manual_seed(1024)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)])
    idx[:, 0] = torch.randint(0, 4, (T,), generator=g)     # four hot experts overflow
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.rand(T, K, generator=g).to(DEV)
    w13, s13, w2, s2 = (t.to(DEV) for t in W.expert_weights(E, H, I, 5, "cpu"))
    buf = api.MoeLayerBuffers(T, E, K, H, I, R, dev)
    y_sep = buf.forward(x, idx.to(DEV), w, w13, s13, w2, s2, fused=False).clone()
    y = buf.forward(x, idx.to(DEV), w, w13, s13, w2, s2).clone()
    pk = api.MoeLayerBuffers(T, E, K, H, I, R, dev, packed=True)
    y_pk = pk.forward(x, idx.to(DEV), w, w13, s13, w2, s2)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16))
    assert torch.equal(y.view(torch.int16), y_pk.view(torch.int16))
    rr = O.route(idx.numpy(), E, R)
    assert np.array_equal(buf.src_map.cpu().numpy(), rr.src_map)
    assert buf.counts.cpu().numpy().tolist() == rr.counts.tolist()
    st = buf.dev_status.cpu().tolist()
    assert st[1] == rr.dropped > 0 and st[0] & api.DEV_CAPACITY_DROPPED
    experts = list(range(0, E, 16))
    wts = host_weights({"w13": w13, "s13": s13, "w2": w2, "s2": s2}, experts)
    src = rr.src_map
    for e in experts:
        tk = np.argwhere((idx.numpy() == e) & (src >= 0))
        if len(tk) == 0:
            continue
        ref = oracle_expert_rows(f32(x[torch.from_numpy(tk[:, 0]).to(DEV)]), wts[e])
        got = f32(buf.out.view(-1, H)[torch.from_numpy(src[tk[:, 0], tk[:, 1]]).long().to(DEV)])
        assert_rows_close(got, ref, what=f"expert {e}")
