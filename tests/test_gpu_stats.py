"""moe_layer_stats against the oracle's byte accounting ("SGLang、NCCL 与 MoE
EP", §5.3: sum over tokens of D_t messages, cross-rank routes) and tile
counting ("SGLang Expert Compute Backend", §5.4: M-blocks and the M-row fill
rate), on the traced scenario (the page's 224 routes, 160 of them cross-rank)
and the decode/prefill/large routings."""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_grouped_topk_gb300 import api
from token_dispatch_grouped_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api._lib.load()
    yield


def _check(idx, E, L, R, src_rank, offsets=None):
    _, counts, _, _ = api.moe_dispatch(torch.zeros(idx.shape[0], 128, dtype=torch.bfloat16, device=DEV),
                                       idx, None, E, R)
    stats = api.moe_layer_stats(idx, counts, L, R, rank_offsets=offsets)
    torch.cuda.synchronize()
    got = api.layer_stats_dict(stats, E, R)
    idx_np = idx.long().cpu().numpy()
    rr = O.route(idx_np, E, R)
    # ids outside [-1, E) are reported and ignored (not routes), so the
    # oracle's accounting sees them as padding
    want = O.route_stats(np.where((idx_np >= 0) & (idx_np < E), idx_np, -1), L, src_rank)
    assert got["valid_routes"] == want["routes"]
    assert got["messages"] == want["messages"]
    assert got["cross_rank_routes"] == want["cross_rank_routes"]
    assert got["kept_routes"] == int(rr.counts.sum())
    assert got["dropped_routes"] == rr.dropped
    assert got["tile_blocks"] == O.m_blocks(rr.counts, 128)
    if got["tile_blocks"]:
        assert abs(got["m_fill_128"] - O.m_fill_rate(rr.counts, 128)) < 1e-12
    assert got["active_experts"] == int((rr.counts > 0).sum())
    assert got["busiest_expert_rows"] == int(rr.counts.max())
    return got


def test_traced_scenario_stats():
    with open(os.path.join(GOLDEN, "traced_scenario.json"), encoding="utf-8") as f:
        g = json.load(f)
    wl = W.WORKLOADS["traced"]
    idx, _ = W.traced_routes(0)
    src = W.source_rank_of_tokens(wl).numpy()
    per = np.array(wl.tokens_per_rank)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(per)]), dtype=torch.int32, device=DEV)
    got = _check(idx.to(DEV), wl.E, wl.L, wl.R, src, offsets)
    assert got["valid_routes"] == g["bytes"]["routes"] == 224
    assert got["cross_rank_routes"] == g["bytes"]["cross_rank_routes"] == 160
    assert got["tile_blocks"] == 4 and got["active_experts"] == 4


@pytest.mark.parametrize("name", ["decode", "prefill", "large"])
def test_synthetic_layer_stats(name):
    """Even token split over the logical ranks (rank_offsets = NULL)."""
    wl = W.WORKLOADS[name]
    idx, _ = W.router(wl.T, wl.E, wl.K, W.router_bias(wl, 0, DEV), 1, DEV)
    src = W.source_rank_of_tokens(wl).numpy()
    got = _check(idx, wl.E, wl.L, wl.R, src)
    assert got["valid_routes"] == wl.T * wl.K


def test_int32_ids_bad_ids_and_empty():
    E, L, R, T, K = 16, 4, 8, 50, 3
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[5, 2] = E + 3                       # invalid: not a route
    src = np.minimum(np.arange(T) // -(-T // (E // L)), E // L - 1)
    _check(idx.to(torch.int32).to(DEV), E, L, R, src)
    empty = _check(torch.empty(0, K, dtype=torch.int64, device=DEV), E, L, R, np.zeros(0, int))
    assert empty["valid_routes"] == 0 and empty["tile_blocks"] == 0
