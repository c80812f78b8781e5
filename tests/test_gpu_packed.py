"""The packed layout ("SGLang Expert Compute Backend", §2.6, compact storage):
expert rows back to back from the prefix of the clamped counts, through
moe_dispatch_packed, moe_expert_compute_packed and moe_combine_packed.

Bit-exact against the oracle's packed source map and against the padded path
(same routing, same arithmetic, only the row addresses differ)."""
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


@pytest.mark.parametrize("T,E,K,R,H", [(300, 33, 5, 40, 640), (4, 8, 2, 4, 256), (2000, 64, 8, 200, 1024),
                                       (0, 6, 2, 10, 256), (257, 9, 3, 1000, 384)])
def test_dispatch_packed_matches_oracle_and_padded(T, E, K, R, H):
    g = torch.Generator().manual_seed(T * 7 + E)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    logits = torch.randn(T, E, generator=g)
    logits[:, : E // 3] += 2.0                      # skew: some experts overflow R
    idx = torch.topk(logits, K, dim=1).indices
    if T > 3:
        idx[3, 0] = -1                              # padding route
    w = torch.rand(T, K, generator=g)
    idx_d, w_d = idx.to(DEV), w.to(DEV)
    recv_p, cnt_p, map_p, st_p = api.moe_dispatch_packed(x, idx_d, w_d, E, R)
    recv_d, cnt_d, map_d, st_d = api.moe_dispatch(x, idx_d, w_d, E, R)
    torch.cuda.synchronize()
    rr = O.route(idx.numpy(), E, R)
    assert cnt_p.cpu().tolist() == rr.counts.tolist() == cnt_d.cpu().tolist()
    assert np.array_equal(map_p.cpu().numpy(), O.packed_src_map(rr.src_map, rr.counts, R))
    assert st_p.cpu().tolist() == st_d.cpu().tolist()
    assert recv_p.shape[0] == api.packed_rows(T, K, E, R)
    off = O.packed_row_offsets(rr.counts)
    for e in range(E):
        c = int(rr.counts[e])
        assert torch.equal(_bits(recv_p[off[e]:off[e] + c]), _bits(recv_d[e, :c])), f"expert {e}"


def _expert_inputs(E, R, H, I, counts, seed):
    g = torch.Generator().manual_seed(seed)
    recv = torch.randn(E, R, H, generator=g).to(torch.bfloat16)
    w13, s13, w2, s2 = W.expert_weights(E, H, I, seed, "cpu")
    return recv, w13.to(DEV), s13.to(DEV), w2.to(DEV), s2.to(DEV)


@pytest.mark.parametrize("E,R,H,I,counts", [
    (4, 384, 512, 384, [300, 129, 0, 17]),
    (13, 256, 384, 256, [1, 31, 32, 33, 63, 64, 65, 127, 129, 192, 193, 256, 0]),
    (3, 200, 256, 128, [200, 199, 64]),
])
def test_expert_compute_packed_matches_padded(E, R, H, I, counts):
    recv, w13, s13, w2, s2 = _expert_inputs(E, R, H, I, counts, seed=21)
    cd = torch.tensor(counts, dtype=torch.int32, device=DEV)
    out_d = api.moe_expert_compute(recv.to(DEV), cd, w13, s13, w2, s2)
    off = O.packed_row_offsets(counts)
    total = int(off[-1])
    rows = total + 37                                     # spare rows must stay untouched
    packed = torch.cat([recv[e, :c] for e, c in enumerate(counts)] +
                       [torch.zeros(rows - total, H, dtype=torch.bfloat16)]).to(DEV)
    out_p = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    api.moe_expert_compute_packed(packed, cd, R, w13, s13, w2, s2, out=out_p, dev_status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0]
    for e, c in enumerate(counts):
        assert torch.equal(_bits(out_p[off[e]:off[e] + c]), _bits(out_d[e, :c])), f"expert {e}"
    assert bool((out_p[total:].float() == 3.0).all()), "rows past the packed range were written"


def test_expert_compute_packed_never_writes_past_rows():
    """Counts that claim more rows than the buffer holds: every row at or past
    `rows` stays untouched (the tail of a larger allocation is a sentinel)."""
    E, R, H, I = 3, 256, 256, 128
    counts = [200, 150, 100]                              # 450 rows claimed
    recv, w13, s13, w2, s2 = _expert_inputs(E, R, H, I, counts, seed=22)
    rows = 300                                            # buffer holds only 300
    big_in = torch.zeros(rows + 200, H, dtype=torch.bfloat16, device=DEV)
    big_in[:rows] = torch.randn(rows, H).to(torch.bfloat16).to(DEV)
    big_out = torch.full((rows + 200, H), 5.0, dtype=torch.bfloat16, device=DEV)
    cd = torch.tensor(counts, dtype=torch.int32, device=DEV)
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    api.moe_expert_compute_packed(big_in[:rows], cd, R, w13, s13, w2, s2, out=big_out[:rows],
                                  dev_status=st)
    torch.cuda.synchronize()
    assert bool((big_out[rows:].float() == 5.0).all())
    assert st.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("name", ["traced", "decode", "prefill"])
def test_layer_packed_bit_identical_to_padded(name):
    d = W.make_layer_inputs(name, seed=0, device=DEV)
    wl = d["wl"]
    dev = torch.device(DEV)
    pad = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    pk = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev, packed=True)
    args = (d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    y_pad = pad.forward(*args, fused=False).clone()
    for fused in (False, True):
        y_pk = pk.forward(*args, fused=fused).clone()
        torch.cuda.synchronize()
        assert torch.equal(_bits(y_pk), _bits(y_pad)), f"fused={fused}"
        assert pk.dev_status.cpu().tolist() == pad.dev_status.cpu().tolist()
    assert pk.recv.shape == (api.packed_rows(wl.T, wl.K, wl.E, wl.R), wl.H)


def test_layer_packed_graph_replay_new_routes():
    """Captured once, replayed with new routings written into the same input
    buffers: the packed lane's output equals the padded lane's each time."""
    d = W.make_layer_inputs("decode", seed=0, device=DEV)
    wl = d["wl"]
    dev = torch.device(DEV)
    pad = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    pk = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev, packed=True)
    x, idx, w = d["x"].clone(), d["topk_idx"].clone(), d["topk_w"].clone()
    wts = (d["w13"], d["s13"], d["w2"], d["s2"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pk.forward(x, idx, w, *wts)                        # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pk.forward(x, idx, w, *wts)
    for seed in (5, 6):
        i2, w2_ = W.router(wl.T, wl.E, wl.K, W.router_bias(wl, seed, DEV), seed + 1, DEV)
        idx.copy_(i2)
        w.copy_(w2_)
        g.replay()
        ref = pad.forward(x, idx, w, *wts)
        torch.cuda.synchronize()
        assert torch.equal(_bits(pk.y), _bits(ref)), f"routing {seed}"


@pytest.mark.parametrize("packed", [False, True])
def test_int32_ids_match_int64_ids(packed):
    """moe_dispatch_ex with int32 router ids: the same counts, slots, payload
    and status as int64 ids, padding routes (-1) and out-of-range ids included."""
    T, E, K, R, H = 500, 16, 4, 100, 384
    g = torch.Generator().manual_seed(31)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    logits = torch.randn(T, E, generator=g)
    logits[:, :3] += 2.5
    idx = torch.topk(logits, K, dim=1).indices
    idx[5, 1] = -1
    idx[7, 0] = E + 3                                     # bad id
    idx[9, 2] = -7                                        # bad id
    w = torch.rand(T, K, generator=g).to(DEV)
    fn = api.moe_dispatch_packed if packed else api.moe_dispatch
    r64 = fn(x, idx.to(DEV), w, E, R)
    r32 = fn(x, idx.to(torch.int32).to(DEV), w, E, R)
    torch.cuda.synchronize()
    for a, b in zip(r64[1:], r32[1:]):                    # counts, src_map, status
        assert torch.equal(a, b)
    counts = r64[1].cpu().tolist()
    if packed:
        total = sum(counts)
        assert torch.equal(_bits(r64[0][:total]), _bits(r32[0][:total]))
    else:
        for e, c in enumerate(counts):                    # capacity rows are never written
            assert torch.equal(_bits(r64[0][e, :c]), _bits(r32[0][e, :c]))
    st = r32[3].cpu().tolist()
    assert st[0] & api.DEV_BAD_EXPERT_ID and st[0] & api.DEV_CAPACITY_DROPPED
    rr = O.route(idx.numpy(), E, R)
    assert r32[1].cpu().tolist() == rr.counts.tolist() and st[1] == rr.dropped


# ------------------------------------------------ interleaved gate/up weights

def _unit_scale_weights(E, H, I, seed):
    """e4m3 codes of both signs (no NaN codes) and one scale for every block,
    so the standard and interleaved layouts describe the same expert."""
    g = torch.Generator().manual_seed(seed)
    def codes(*shape):
        c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(torch.uint8)
        c[(c & 0x7F) == 0x7F] = 0
        return c
    w13, w2 = codes(E, 2 * I, H), codes(E, H, I)
    s13 = torch.full((E, 2 * I // 128, H // 128), 1e-3)
    s2 = torch.full((E, H // 128, I // 128), 2e-3)
    return w13, s13, w2, s2


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("shape", [(112, 8, 2, 256, 128, 128), (600, 16, 4, 512, 384, 256)])
def test_interleaved_w13_bit_identical_to_standard(packed, shape):
    """Uniform block scales: interleaving W13's rows (2j gate, 2j+1 up) and
    flagging MOE_W13_INTERLEAVED gives the standard layer's bytes, through
    moe_expert_compute and through the fused dispatch+quant path."""
    T, E, K, H, I, R = shape
    w13, s13, w2, s2 = _unit_scale_weights(E, H, I, seed=41)
    inter = torch.empty_like(w13)
    inter[:, 0::2], inter[:, 1::2] = w13[:, :I], w13[:, I:]
    dev = torch.device(DEV)
    g = torch.Generator().manual_seed(42)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    idx = torch.topk(torch.randn(T, E, generator=g), K, dim=1).indices.to(DEV)
    w = torch.rand(T, K, generator=g).to(DEV)
    std = api.MoeLayerBuffers(T, E, K, H, I, R, dev, packed=packed)
    itl = api.MoeLayerBuffers(T, E, K, H, I, R, dev, packed=packed, w13_interleaved=True)
    args = (x, idx, w)
    y_std = std.forward(*args, w13.to(DEV), s13.to(DEV), w2.to(DEV), s2.to(DEV), fused=False).clone()
    y_itl = itl.forward(*args, inter.to(DEV), s13.to(DEV), w2.to(DEV), s2.to(DEV), fused=False).clone()
    torch.cuda.synchronize()
    assert torch.equal(_bits(y_itl), _bits(y_std))
    assert float(y_std.float().abs().max()) > 0
    # the fused dispatch+quant path hands the flag to moe_gemm_gateup_down
    y_fused = itl.forward(*args, inter.to(DEV), s13.to(DEV), w2.to(DEV), s2.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(_bits(y_fused), _bits(y_std))


def test_interleaved_w13_matches_oracle():
    """Block-scaled interleaved weights (each 128x128 block of the interleaved
    layout with its own scale) against the oracle's interleaved expert."""
    E, R, H, I = 3, 256, 512, 256
    counts = [200, 70, 13]
    g = torch.Generator().manual_seed(43)
    recv = torch.randn(E, R, H, generator=g).to(torch.bfloat16)
    w13, s13, w2, s2 = W.expert_weights(E, H, I, 44, "cpu")   # read as interleaved rows
    cd = torch.tensor(counts, dtype=torch.int32, device=DEV)
    out = api.moe_expert_compute(recv.to(DEV), cd, w13.to(DEV), s13.to(DEV), w2.to(DEV), s2.to(DEV),
                                 w13_interleaved=True)
    torch.cuda.synchronize()
    from helpers import assert_rows_close, f32, u8
    for e, c in enumerate(counts):
        xq, sx = O.quantize_rows(f32(recv[e, :c]))
        ref, _, _, _ = O.expert_forward(xq, sx, u8(w13[e]), f32(s13[e]), u8(w2[e]), f32(s2[e]),
                                        interleaved=True)
        assert_rows_close(f32(out[e, :c]), ref, what=f"expert {e}")


@pytest.mark.parametrize("bits,packed", [(32, False), (64, True), (32, True)])
def test_dispatch_quant_ex_variants(bits, packed):
    """moe_dispatch_quant_ex with int32 ids and/or the packed layout: the
    source map is the oracle's (packed: its packed map), and every kept row
    holds the oracle's e4m3 codes and scales of its token row."""
    T, E, K, R, H = 700, 24, 6, 150, 512
    g = torch.Generator().manual_seed(41 + bits + packed)
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[:, 0] = torch.randint(0, 3, (T,), generator=g)      # hot experts overflow R
    idx[4, 1] = E + 2                                        # invalid id
    x = (torch.randn(T, H, generator=g) * torch.rand(T, 1, generator=g) * 4).to(torch.bfloat16)
    rows = api.packed_rows(T, K, E, R) if packed else 0
    xd = x.to(DEV)
    idd = idx.to(DEV).to(torch.int32 if bits == 32 else torch.int64)
    xq, xs, counts, src, st = api.moe_dispatch_quant(xd, idd, None, E, R, rows=rows)
    torch.cuda.synchronize()
    rr = O.route(idx.numpy(), E, R)
    want_map = O.packed_src_map(rr.src_map, rr.counts, R) if packed else rr.src_map
    assert counts.cpu().numpy().tolist() == rr.counts.tolist()
    assert np.array_equal(src.cpu().numpy(), want_map)
    stv = st.cpu().tolist()
    assert stv[1] == rr.dropped and bool(stv[0] & api.DEV_BAD_EXPERT_ID)
    keep = want_map >= 0
    q = torch.from_numpy(want_map[keep]).long()
    tok = np.nonzero(keep)[0]
    codes, scales = O.quantize_rows(x.float().numpy()[tok])
    assert np.array_equal(xq.view(-1, H).cpu()[q].numpy(), codes)
    assert np.array_equal(xs.view(-1, H // 128).cpu()[q].numpy(), scales)


@pytest.mark.parametrize("name,packed,bits", [("traced", True, 64), ("decode", True, 32),
                                              ("prefill", True, 64), ("decode", False, 32)])
def test_layer_fused_path_every_variant(name, packed, bits):
    """The fused dispatch+quant layer path on packed lanes and int32 ids is
    bit-identical to the unfused padded path."""
    d = W.make_layer_inputs(name, seed=8, device=DEV)
    wl = d["wl"]
    dev = torch.device(DEV)
    ids = d["topk_idx"].to(torch.int32) if bits == 32 else d["topk_idx"]
    wts = (d["w13"], d["s13"], d["w2"], d["s2"])
    ref = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    y_ref = ref.forward(d["x"], d["topk_idx"], d["topk_w"], *wts, fused=False).clone()
    lane = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev, packed=packed)
    y = lane.forward_fused(d["x"], ids, d["topk_w"], *wts)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(y_ref))
    assert lane.dev_status.cpu().tolist() == ref.dev_status.cpu().tolist()
