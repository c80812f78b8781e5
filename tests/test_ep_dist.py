"""The expert-parallel layer's exchange logic on two gloo ranks (CPU).

ExpertParallelLayer.forward runs as in a multi-GPU job -- send counts, the
payload and route-list all-to-alls, the return splits read from the route
offsets, the returned rows and flags -- with the per-phase kernel calls stood
in by plain CPU code written here from the calls' documented contracts
(include/moe.h, expert parallelism) on top of the oracle's routing and expert
math.  The y each rank returns must equal, bit for bit, the same stand-in
arithmetic run on all ranks' tokens in one process ("SGLang、NCCL 与 MoE EP",
§2.3.2 dedup per destination rank, §3.2 results back into the source's route
slots), with capacity drops at the destinations."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from token_dispatch_grouped_topk_gb300 import ep
from token_dispatch_grouped_topk_gb300 import workloads as W

E, L, K, H, I, R = 8, 4, 3, 128, 128, 6
T_RANK = (11, 14)


def _bf16(a):
    return O.f32_to_bf16_rne(np.asarray(a, np.float32))


class OracleEpOps:
    """CPU stand-ins for the phases of a rank's data path."""

    def __init__(self, weights):
        self.weights = weights   # this rank's experts: (w13 [L,2I,H], s13, w2, s2) numpy

    def pack(self, x, topk_idx, E_, L_):
        idx = topk_idx.numpy()
        T = idx.shape[0]
        Wr = E_ // L_
        rows = [[] for _ in range(Wr)]           # per destination: (t, route list)
        owner = {}
        for t in range(T):
            for k in range(K):
                e = int(idx[t, k])
                if not 0 <= e < E_:
                    continue
                d = e // L_
                if (t, d) not in owner:
                    owner[(t, d)] = len(rows[d])
                    rows[d].append((t, [int(idx[t, j]) % L_ if 0 <= idx[t, j] < E_ and idx[t, j] // L_ == d
                                        else -1 for j in range(K)]))
        base = np.cumsum([0] + [len(r) for r in rows])
        S = int(base[-1])
        send_x = torch.zeros(max(S, 1), H, dtype=torch.bfloat16)
        send_ids = torch.full((max(S, 1), K), -1, dtype=torch.int32)
        route_msg = torch.full((T, K), -1, dtype=torch.int32)
        route_pos = torch.full((T, K), -1, dtype=torch.int32)
        for d in range(Wr):
            for i, (t, ids) in enumerate(rows[d]):
                u = int(base[d]) + i
                send_x[u] = x[t]
                send_ids[u] = torch.tensor(ids, dtype=torch.int32)
                p = 0
                for k in range(K):
                    if ids[k] >= 0:
                        route_msg[t, k], route_pos[t, k] = u, p
                        p += 1
        return {"send_x": send_x, "send_ids": send_ids,
                "send_counts": torch.tensor([len(r) for r in rows], dtype=torch.int32),
                "route_msg": route_msg, "route_pos": route_pos, "status": torch.zeros(2, dtype=torch.int32)}

    def local(self, recv_x, recv_ids, L_, R_, weights, gemm_launch=None):
        ids = recv_ids.numpy()
        rr = O.route(ids, L_, R_)
        xs = recv_x.float().numpy()
        out = np.zeros((L_ * R_, H), np.float32)
        for e in range(L_):
            tk = np.argwhere((ids == e) & (rr.src_map >= 0))
            if len(tk) == 0:
                continue
            xq, sx = O.quantize_rows(xs[tk[:, 0]])
            w13, s13, w2, s2 = (w[e] for w in self.weights)
            out[rr.src_map[tk[:, 0], tk[:, 1]]] = _bf16(O.expert_forward(xq, sx, w13, s13, w2, s2)[0])
        st = torch.tensor([0, rr.dropped], dtype=torch.int32)
        return {"out": torch.from_numpy(out).to(torch.bfloat16), "src_map": torch.from_numpy(rr.src_map),
                "counts": torch.from_numpy(rr.counts), "status": st}

    def offsets(self, ids):
        n = (ids >= 0).sum(dim=1).to(torch.int32)
        return torch.cat([torch.zeros(1, dtype=torch.int32), torch.cumsum(n, 0).to(torch.int32)])

    def ret(self, out, src_map, ids, offsets, n_ret):
        ret_x = torch.zeros(n_ret, H, dtype=torch.bfloat16)
        flag = torch.zeros(n_ret, dtype=torch.int32)
        for j in range(ids.shape[0]):
            p = 0
            for k in range(K):
                if ids[j, k] < 0:
                    continue
                r = int(offsets[j]) + p
                p += 1
                q = int(src_map[j, k])
                if q >= 0:
                    ret_x[r] = out[q]
                    flag[r] = 1
        return ret_x, flag

    def result(self, route_msg, route_pos, offsets, flag, n_ret):
        rm = torch.full_like(route_msg, -1)
        for (t, k), u in np.ndenumerate(route_msg.numpy()):
            if u >= 0:
                r = int(offsets[u]) + int(route_pos[t, k])
                if r < n_ret and flag[r]:
                    rm[t, k] = r
        return rm

    def combine(self, ret_x, result_map, topk_w, T, H_):
        return torch.from_numpy(O.combine_f32_sequential(ret_x.float().numpy(), result_map.numpy(),
                                                         topk_w.numpy())).to(torch.bfloat16)


def _inputs():
    g = torch.Generator().manual_seed(21)
    T = sum(T_RANK)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)])
    idx[:, 0] = torch.randint(0, 2, (T,), generator=g)     # experts 0 and 1 overflow R
    idx[3, 2] = -1
    w = torch.rand(T, K, generator=g)
    w13, s13, w2, s2 = (t.numpy() for t in W.expert_weights(E, H, I, 5, "cpu"))
    return x, idx, w, (w13, s13, w2, s2)


def _single_process_reference(x, idx, w, weights):
    """The same stand-in arithmetic on all tokens at once: canonical routing
    with capacity R per expert, expert outputs rounded to BF16, fp32 combine."""
    rr = O.route(idx.numpy(), E, R)
    xs = x.float().numpy()
    out = np.zeros((E * R, H), np.float32)
    for e in range(E):
        tk = np.argwhere((idx.numpy() == e) & (rr.src_map >= 0))
        if len(tk) == 0:
            continue
        xq, sx = O.quantize_rows(xs[tk[:, 0]])
        out[rr.src_map[tk[:, 0], tk[:, 1]]] = _bf16(O.expert_forward(xq, sx, *(wt[e] for wt in weights))[0])
    return O.combine_f32_sequential(out, rr.src_map, w.numpy()), rr


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, idx, w, weights = _inputs()
        t0 = sum(T_RANK[:rank])
        sl = slice(t0, t0 + T_RANK[rank])
        mine = tuple(wt[rank * L:(rank + 1) * L] for wt in weights)
        layer = ep.ExpertParallelLayer(E, L, R, rank, comm=ep.TorchDistComm(), ops=OracleEpOps(mine))
        res = layer.forward(x[sl], idx[sl], w[sl], *mine)
        q.put((rank, res.y.float().numpy(), res.send_counts, res.recv_counts,
               int(res.local_status[1])))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_equal_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict((item[0], item[1:]) for item in (q.get(timeout=300) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x, idx, w, weights = _inputs()
    y_ref, rr = _single_process_reference(x, idx, w, weights)
    assert rr.dropped > 0
    y = np.concatenate([got[0][0], got[1][0]])
    assert np.array_equal(y, y_ref)
    # one message per (token, destination rank), and what one rank sends the other receives
    assert got[0][1][1] == got[1][2][0] and got[1][1][0] == got[0][2][1]
    dest_sets = [len({int(e) // L for e in row if e >= 0}) for row in idx.numpy()]
    assert sum(got[0][1]) + sum(got[1][1]) == sum(dest_sets)
    # the destinations' capacity drops are the one-process drops
    assert got[0][3] + got[1][3] == rr.dropped
