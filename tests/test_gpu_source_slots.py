"""The per-source fixed-slot receive layout ("DeepEP 架构与实现笔记", §9.5)
through moe_dispatch_source_slots / moe_expert_compute_source_slots (BF16
slots) and moe_dispatch_quant_source_slots / moe_gemm_source_slots (FP8 slots).

Dispatch bit-exact against the oracle's route_source_slots (source map,
per-expert and per-(expert, source) counts, drops, bad ids, payload rows), the
FP8 slots against the oracle's quantisation of each token row; expert outputs
and the layer output bit-identical to the padded layout on the same routes (a
row's arithmetic does not depend on where the row sits) and between the BF16
and FP8 slot paths; rows between the source ranges never written."""
import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_grouped_topk_gb300 import api
from token_dispatch_grouped_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api._lib.load()
    yield
    torch.cuda.synchronize()


def _bits(t):
    return t.view(torch.int16)


def _src_rank(T, Wr, offsets):
    if offsets is None:
        per = -(-T // Wr)
        return np.minimum(np.arange(T) // max(per, 1), Wr - 1)
    return np.searchsorted(np.asarray(offsets), np.arange(T), side="right") - 1


def _check_dispatch(x, idx, E, L, mt, offsets=None):
    T, H = x.shape
    Wr = E // L
    off_d = None if offsets is None else torch.tensor(offsets, dtype=torch.int32, device=DEV)
    recv = torch.full((E, Wr * mt, H), 5.0, dtype=torch.bfloat16, device=DEV)
    recv, counts, seg, src, st = api.moe_dispatch_source_slots(x.to(DEV), idx.to(DEV), None, E, L, mt,
                                                               rank_offsets=off_d, recv=recv)
    torch.cuda.synchronize()
    res = O.route_source_slots(idx.long().numpy(), E, L, mt, _src_rank(T, Wr, offsets))
    assert np.array_equal(src.cpu().numpy(), res.src_map)
    assert counts.cpu().numpy().tolist() == res.counts.tolist()
    assert np.array_equal(seg.cpu().numpy(), res.seg_counts)
    stv = st.cpu().tolist()
    assert stv[1] == res.dropped
    assert bool(stv[0] & api.DEV_CAPACITY_DROPPED) == (res.dropped > 0)
    assert bool(stv[0] & api.DEV_BAD_EXPERT_ID) == res.bad_id
    flat = recv.view(-1, H)
    keep = res.src_map >= 0
    q = torch.from_numpy(res.src_map[keep]).long().to(DEV)
    tok = torch.from_numpy(np.nonzero(keep)[0]).long().to(DEV)
    assert torch.equal(_bits(flat[q]), _bits(x.to(DEV)[tok]))
    written = torch.zeros(flat.shape[0], dtype=torch.bool, device=DEV)
    written[q] = True
    assert bool((flat[~written] == 5.0).all()), "rows between the source ranges were written"
    return res, recv, counts, seg, src


def _check_dispatch_fp8(x, idx, E, L, mt, offsets=None, max_tokens=512):
    """moe_dispatch_quant_source_slots: routing outputs equal to the BF16 slot
    dispatch's (itself checked against the oracle); each kept slot holds the
    oracle's e4m3 codes and scales of its token row; other rows untouched."""
    T, H = x.shape
    G = H // 128
    Wr = E // L
    res, recv, counts, seg, src = _check_dispatch(x, idx, E, L, mt, offsets)
    off_d = None if offsets is None else torch.tensor(offsets, dtype=torch.int32, device=DEV)
    xq = torch.full((E, Wr * mt, H), 0x5A, dtype=torch.uint8, device=DEV)
    xs = torch.full((E, Wr * mt, G), -3.0, dtype=torch.float32, device=DEV)
    xq, xs, c8, seg8, src8, st8 = api.moe_dispatch_quant_source_slots(
        x.to(DEV), idx.to(DEV), None, E, L, mt, rank_offsets=off_d, xq=xq, xs=xs)
    torch.cuda.synchronize()
    assert torch.equal(c8, counts) and torch.equal(seg8, seg) and torch.equal(src8, src)
    stv = st8.cpu().tolist()
    assert stv[1] == res.dropped
    assert bool(stv[0] & api.DEV_CAPACITY_DROPPED) == (res.dropped > 0)
    assert bool(stv[0] & api.DEV_BAD_EXPERT_ID) == res.bad_id
    q_rows, s_rows = xq.view(-1, H), xs.view(-1, G)
    keep = res.src_map >= 0
    slots = torch.from_numpy(res.src_map[keep]).long().to(DEV)
    tok = np.nonzero(keep)[0]
    written = torch.zeros(q_rows.shape[0], dtype=torch.bool, device=DEV)
    written[slots] = True
    assert bool((q_rows[~written] == 0x5A).all()) and bool((s_rows[~written] == -3.0).all())
    # every slot of a token holds the same codes; the oracle's on a sample of tokens
    first = {}
    for t, sl in zip(tok.tolist(), res.src_map[keep].tolist()):
        first.setdefault(t, sl)
    firsts = torch.tensor([first[t] for t in tok.tolist()], dtype=torch.long, device=DEV)
    assert torch.equal(q_rows[slots], q_rows[firsts]) and torch.equal(s_rows[slots], s_rows[firsts])
    has = np.array(sorted(first))
    if len(has) > max_tokens:
        has = np.sort(np.random.default_rng(0).choice(has, max_tokens, replace=False))
    if len(has):
        codes, scales = O.quantize_rows(x[torch.from_numpy(has)].float().cpu().numpy())
        rows = torch.tensor([first[t] for t in has.tolist()], dtype=torch.long, device=DEV)
        assert np.array_equal(q_rows[rows].cpu().numpy(), codes)
        assert np.array_equal(s_rows[rows].cpu().numpy(), scales)
    return res, xq, xs, seg, src, recv


@pytest.mark.parametrize("bits", [64, 32])
def test_dispatch_random_with_drops_and_empty_ranks(bits):
    E, L, K, mt, H = 40, 5, 4, 3, 256
    Wr = E // L
    g = torch.Generator().manual_seed(3 + bits)
    T = 150
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[:, 0] = torch.randint(0, 3, (T,), generator=g)      # hot experts overflow each source range
    idx[7, 2] = E + 5                                         # invalid id
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    offsets = [0, 0, 20, 20, 61, 100, 100, 140, 150]           # ranks 0, 2 and 5 send nothing
    assert len(offsets) == Wr + 1
    ids = idx.to(torch.int32) if bits == 32 else idx
    res, *_ = _check_dispatch(x, ids, E, L, mt, offsets)
    assert res.dropped > 0 and res.bad_id
    res2, *_ = _check_dispatch(x, ids, E, L, mt, None)     # even split
    assert res2.dropped > 0


@pytest.mark.parametrize("bits", [64, 32])
@pytest.mark.parametrize("E,L,K,mt,H,T", [(40, 5, 4, 3, 256, 150), (12, 3, 4, 50, 1152, 300),
                                          (256, 8, 8, 32, 7168, 256), (16, 16, 2, 7, 128, 1),
                                          (8, 2, 3, 5, 384, 0), (64, 8, 32, 4, 256, 40),
                                          (16, 4, 1, 10, 512, 100)])
def test_dispatch_quant_source_slots(bits, E, L, K, mt, H, T):
    """FP8 slots: drops, an invalid id, ranks that send nothing, one group per
    row, a ragged last pass of groups (9 groups), the decode layer's shape, one
    token and no tokens, top-32 (one token per warp) and top-1 (32 tokens per
    warp)."""
    Wr = E // L
    g = torch.Generator().manual_seed(E + H + T + bits)
    idx = torch.randint(-1, E, (T, K), generator=g)
    if T > 1:
        idx[:, 0] = torch.randint(0, 3, (T,), generator=g)
        idx[T // 2, K - 1] = E + 5
    x = (torch.randn(T, H, generator=g) * 3).to(torch.bfloat16)
    if T > 2:
        x[1, :128] = 0                                    # an all-zero group
    offsets = None
    if T >= Wr:
        cuts = np.sort(np.random.default_rng(T).integers(0, T + 1, Wr - 1))
        offsets = [0] + cuts.tolist() + [T]
    ids = idx.to(torch.int32) if bits == 32 else idx
    _check_dispatch_fp8(x, ids, E, L, mt, offsets)
    _check_dispatch_fp8(x, ids, E, L, mt, None)


def test_dispatch_traced_scenario_pins():
    """Traced scenario with the pages' per-rank slot count C = 64: E0 gets 16,
    31 and 64 rows in the ranges of source ranks 1, 2 and 3."""
    wl = W.WORKLOADS["traced"]
    idx, _ = W.traced_routes(0)
    x = W.activations(wl.T, wl.H, 2)
    offsets = np.concatenate([[0], np.cumsum(wl.tokens_per_rank)]).tolist()
    res, _, counts, seg, src = _check_dispatch(x, idx, wl.E, wl.L, 64, offsets)
    assert seg[0].cpu().tolist() == [0, 16, 31, 64]
    assert counts.cpu().tolist() == [111, 1, 0, 0, 0, 0, 1, 111]
    assert src[21].cpu().tolist() == [1 * 256 + 2 * 64, 6 * 256 + 2 * 64]


@pytest.mark.parametrize("name,mt", [("decode", 32), ("traced", 64)])
def test_layer_source_slots_equals_padded(name, mt):
    """Whole layer on the per-source layout, on its default path (FP8 slots)
    and on the BF16 slots: every kept route's expert output and y
    bit-identical to the padded layout's and between the two paths, out rows
    between the source ranges untouched.  Decode: 8 ranks x 32 tokens, so
    W * max_tokens = 256 = the decode capacity and nothing is dropped."""
    d = W.make_layer_inputs(name, seed=1, device=DEV)
    wl = d["wl"]
    dev = torch.device(DEV)
    Wr = wl.E // wl.L
    offsets = None
    if wl.tokens_per_rank:
        offsets = torch.tensor(np.concatenate([[0], np.cumsum(wl.tokens_per_rank)]), dtype=torch.int32,
                               device=DEV)
    ss = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, Wr * mt, dev, source_slots=mt, L=wl.L,
                             rank_offsets=offsets)
    ss.out.fill_(7.0)
    pad = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, Wr * mt, dev)
    args = (d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    y_ss = ss.forward(*args).clone()
    out_fused = ss.out.clone()
    assert ss._recv is None, "the default path formed the BF16 slots"
    ss.out.fill_(7.0)
    y_sep = ss.forward(*args, fused=False).clone()
    y_pad = pad.forward(*args).clone()
    torch.cuda.synchronize()
    assert torch.equal(_bits(y_sep), _bits(y_ss))
    assert torch.equal(_bits(ss.out), _bits(out_fused))
    assert ss.dev_status.cpu().tolist() == pad.dev_status.cpu().tolist() == [0, 0]
    assert torch.equal(ss.counts, pad.counts)
    sm_ss, sm_pad = ss.src_map.cpu().numpy(), pad.src_map.cpu().numpy()
    keep = sm_ss >= 0
    assert np.array_equal(keep, sm_pad >= 0)
    H = wl.H
    a = ss.out.view(-1, H)[torch.from_numpy(sm_ss[keep]).long().to(DEV)]
    b = pad.out.view(-1, H)[torch.from_numpy(sm_pad[keep]).long().to(DEV)]
    assert torch.equal(_bits(a), _bits(b))
    assert torch.equal(_bits(y_ss), _bits(y_pad))
    written = torch.zeros(ss.out.view(-1, H).shape[0], dtype=torch.bool, device=DEV)
    written[torch.from_numpy(sm_ss[keep]).long().to(DEV)] = True
    assert bool((ss.out.view(-1, H)[~written] == 7.0).all()), "gap rows of out were written"


def test_expert_compute_source_slots_both_launch_forms():
    """The per-source layout's expert compute, one launch and two launches,
    with blocks that hold only gaps and ranges cut short by drops; the GEMMs on
    the FP8 slots (moe_gemm_source_slots) give the same output, bit for bit."""
    E, L, K, mt, H, I, T = 12, 3, 4, 50, 512, 256, 300
    g = torch.Generator().manual_seed(17)
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[:, 0] = torch.randint(0, 2, (T,), generator=g)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    res, recv, counts, seg, src = _check_dispatch(x, idx, E, L, mt)
    w13, s13, w2, s2 = (t.to(DEV) for t in W.expert_weights(E, H, I, 4, "cpu"))
    outs = []
    for form in ("one", "two"):
        out = torch.full_like(recv, 9.0)
        st = torch.zeros(2, dtype=torch.int32, device=DEV)
        api.moe_expert_compute_source_slots(recv, counts, seg, L, mt, w13, s13, w2, s2, out=out,
                                            dev_status=st, gemm_launch=form)
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, 0]
        outs.append(out)
    assert torch.equal(_bits(outs[0]), _bits(outs[1]))
    _, xq, xs, seg8, _, _ = _check_dispatch_fp8(x, idx, E, L, mt)
    assert torch.equal(seg8, seg)
    for form in ("one", "two"):
        out = torch.full_like(recv, 9.0)
        st = torch.zeros(2, dtype=torch.int32, device=DEV)
        api.moe_gemm_source_slots(xq, xs, seg8, L, mt, w13, s13, w2, s2, out=out, dev_status=st,
                                  gemm_launch=form)
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, 0]
        assert torch.equal(_bits(out), _bits(outs[0])), form
    keep = res.src_map >= 0
    flat = outs[0].view(-1, H)
    q = torch.from_numpy(res.src_map[keep]).long().to(DEV)
    written = torch.zeros(flat.shape[0], dtype=torch.bool, device=DEV)
    written[q] = True
    assert bool((flat[~written] == 9.0).all())
    # against the padded path on the same rows (canonical routing, R = W * mt)
    R = (E // L) * mt
    rp, cp, mp, _ = api.moe_dispatch(x.to(DEV), idx.to(DEV), None, E, R)
    outp = api.moe_expert_compute(rp, cp, w13, s13, w2, s2)
    torch.cuda.synchronize()
    mp = mp.cpu().numpy()
    both = keep & (mp >= 0)
    a = flat[torch.from_numpy(res.src_map[both]).long().to(DEV)]
    b = outp.view(-1, H)[torch.from_numpy(mp[both]).long().to(DEV)]
    assert torch.equal(_bits(a), _bits(b))
    # interleaved W13 rows: the BF16 and FP8 slot paths agree with each other
    inter = []
    for fp8 in (False, True):
        out = torch.full_like(recv, 9.0)
        st = torch.zeros(2, dtype=torch.int32, device=DEV)
        if fp8:
            api.moe_gemm_source_slots(xq, xs, seg8, L, mt, w13, s13, w2, s2, out=out,
                                      dev_status=st, w13_interleaved=True)
        else:
            api.moe_expert_compute_source_slots(recv, counts, seg, L, mt, w13, s13, w2, s2,
                                                out=out, dev_status=st, w13_interleaved=True)
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, 0]
        inter.append(out)
    assert torch.equal(_bits(inter[0]), _bits(inter[1]))
    assert not torch.equal(_bits(inter[0]), _bits(outs[0]))   # the flag reaches the GEMM


@pytest.mark.parametrize("fused", [True, False])
def test_layer_source_slots_degenerate(fused):
    """The per-source lane on no tokens (counts and seg_counts reset) and on
    every route a padding route (no slot rows, y = 0), on both paths."""
    E, L, K, H, I, mt = 8, 2, 2, 256, 128, 6
    Wr = E // L
    dev = torch.device(DEV)
    w13, s13, w2, s2 = (t.to(DEV) for t in W.expert_weights(E, H, I, 3, "cpu"))
    ss = api.MoeLayerBuffers(0, E, K, H, I, Wr * mt, dev, source_slots=mt, L=L)
    ss.counts.fill_(99)
    ss.seg_counts.fill_(99)
    y = ss.forward(torch.empty(0, H, dtype=torch.bfloat16, device=DEV),
                   torch.empty(0, K, dtype=torch.int64, device=DEV), torch.empty(0, K, device=DEV),
                   w13, s13, w2, s2, fused=fused)
    torch.cuda.synchronize()
    assert y.shape == (0, H)
    assert ss.counts.cpu().tolist() == [0] * E
    assert bool((ss.seg_counts == 0).all()) and ss.dev_status.cpu().tolist() == [0, 0]
    T = 20
    g = torch.Generator().manual_seed(5)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    ss = api.MoeLayerBuffers(T, E, K, H, I, Wr * mt, dev, source_slots=mt, L=L)
    ss.y.fill_(7.0)
    ss.out.fill_(9.0)
    y = ss.forward(x, torch.full((T, K), -1, dtype=torch.int64, device=DEV),
                   torch.rand(T, K, generator=g).to(DEV), w13, s13, w2, s2, fused=fused)
    torch.cuda.synchronize()
    assert ss.counts.cpu().tolist() == [0] * E and bool((ss.seg_counts == 0).all())
    assert bool((y.float() == 0).all()) and bool((ss.src_map == -1).all())
    assert bool((ss.out.float() == 9.0).all()), "no slot row may be written"
