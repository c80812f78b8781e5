"""The expert-parallel layer's CUDA data path (moe_ep_pack, the local layer,
moe_ep_route_offsets, moe_ep_return, moe_ep_result_map, moe_combine_packed)
against the one-GPU layer on all ranks' tokens, bit for bit.

W ranks are emulated on one GPU as W host threads, each running
ExpertParallelLayer.forward for its own tokens and experts; their all-to-alls
meet at a host barrier and move rows with device copies.  No kernel waits on
another rank's kernel.  A one-rank NCCL process group runs the same forward
through torch.distributed."""
import os
import socket
import threading

import numpy as np
import pytest
import torch

from token_dispatch_grouped_topk_gb300 import api, ep
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


class _Shared:
    def __init__(self, world):
        self.world = world
        self.slots = [None] * world
        self.barrier = threading.Barrier(world, timeout=120)


class ThreadComm:
    """All-to-all between rank threads of one process: each deposits its send
    tensor and splits, then copies its chunk from every other rank's tensor."""

    def __init__(self, shared, rank):
        self.s, self.rank = shared, rank

    def all_to_all(self, out, inp, out_splits, in_splits):
        torch.cuda.current_stream().synchronize()
        self.s.slots[self.rank] = (inp, list(in_splits))
        self.s.barrier.wait()
        off = 0
        for src in range(self.s.world):
            t, sp = self.s.slots[src]
            start, n = sum(sp[:self.rank]), sp[self.rank]
            assert n == out_splits[src]
            if n:
                out[off:off + n].copy_(t[start:start + n])
            off += n
        torch.cuda.current_stream().synchronize()
        self.s.barrier.wait()


def _run_ranks(world, E, R, x, idx, w, weights, tokens_per_rank, gemm_launch=None):
    L = E // world
    shared = _Shared(world)
    results, errors = [None] * world, []

    def body(r):
        try:
            t0 = sum(tokens_per_rank[:r])
            sl = slice(t0, t0 + tokens_per_rank[r])
            mine = tuple(wt[r * L:(r + 1) * L].contiguous() for wt in weights)
            layer = ep.ExpertParallelLayer(E, L, R, r, comm=ThreadComm(shared, r), gemm_launch=gemm_launch)
            results[r] = layer.forward(x[sl].contiguous(), idx[sl].contiguous(), w[sl].contiguous(), *mine)
            torch.cuda.current_stream().synchronize()
        except BaseException as exc:   # surfaced below
            errors.append(exc)
            shared.barrier.abort()

    threads = [threading.Thread(target=body, args=(r,)) for r in range(world)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    if errors:
        raise errors[0]
    return results


@pytest.mark.parametrize("name,world", [("decode", 2), ("decode", 8), ("traced", 4)])
def test_emulated_ranks_equal_one_gpu_layer(name, world):
    """decode: 8 ranks x 8 experts, 32 tokens each (and the same experts over
    2 ranks); traced: the pages' 4 ranks with [0, 16, 32, 64] tokens."""
    d = W.make_layer_inputs(name, seed=3, device=DEV)
    wl = d["wl"]
    T = wl.T
    per = list(wl.tokens_per_rank) if (wl.tokens_per_rank and world == wl.W) else \
        [T // world + (1 if r < T % world else 0) for r in range(world)]
    weights = (d["w13"], d["s13"], d["w2"], d["s2"])
    one = api.MoeLayerBuffers(T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    y_ref = one.forward(d["x"], d["topk_idx"], d["topk_w"], *weights).clone()
    torch.cuda.synchronize()
    res = _run_ranks(world, wl.E, wl.R, d["x"], d["topk_idx"], d["topk_w"], weights, per)
    y = torch.cat([r.y for r in res])
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    L = wl.E // world
    local = torch.cat([r.local_counts for r in res])
    assert torch.equal(local, one.counts)
    assert sum(int(r.local_status[1]) for r in res) == int(one.dev_status[1])
    # one message per (token, destination rank)
    idx = d["topk_idx"].cpu().numpy()
    assert sum(sum(r.send_counts) for r in res) == sum(len({int(e) // L for e in row if e >= 0}) for row in idx)


def test_emulated_ranks_with_capacity_drops_and_bad_ids():
    """Skewed routing that overflows R at the destinations, padding routes and
    an out-of-range id; both GEMM launch forms."""
    E, K, H, I, R, world = 16, 4, 512, 256, 24, 4
    g = torch.Generator().manual_seed(8)
    per = [40, 0, 57, 23]                     # rank 1 has no tokens
    T = sum(per)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)])
    idx[:, 0] = torch.randint(0, 2, (T,), generator=g)
    idx[idx == 5] = -1
    idx[7, 1] = E + 3
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    idx, w = idx.to(DEV), torch.rand(T, K, generator=g).to(DEV)
    weights = tuple(t.to(DEV) for t in W.expert_weights(E, H, I, 6, "cpu"))
    one = api.MoeLayerBuffers(T, E, K, H, I, R, torch.device(DEV))
    y_ref = one.forward(x, idx, w, *weights).clone()
    torch.cuda.synchronize()
    assert int(one.dev_status[1]) > 0
    for form in ("one", "two"):
        res = _run_ranks(world, E, R, x, idx, w, weights, per, gemm_launch=form)
        y = torch.cat([r.y for r in res])
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), form
        assert sum(int(r.local_status[1]) for r in res) == int(one.dev_status[1])
        assert any(int(r.source_status[0]) & api.DEV_BAD_EXPERT_ID for r in res)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_one_rank_nccl_group():
    """The forward through torch.distributed (NCCL) on a one-rank group: the
    all-to-alls are identities and y equals the one-GPU layer."""
    import torch.distributed as dist
    d = W.make_layer_inputs("traced", seed=5, device=DEV)
    wl = d["wl"]
    weights = (d["w13"], d["s13"], d["w2"], d["s2"])
    one = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    y_ref = one.forward(d["x"], d["topk_idx"], d["topk_w"], *weights).clone()
    torch.cuda.synchronize()
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=torch.device(DEV, torch.cuda.current_device()))
    try:
        layer = ep.ExpertParallelLayer(wl.E, wl.E, wl.R, 0, comm=ep.TorchDistComm())
        res = layer.forward(d["x"], d["topk_idx"], d["topk_w"], *weights)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert torch.equal(res.y.view(torch.int16), y_ref.view(torch.int16))
