"""Expert parallelism across ranks: one MoE layer whose E experts are split
over W ranks (rank r holds experts [r*L, r*L + L)), each rank with its own
tokens, exchanging token rows and expert outputs with all-to-alls.

"SGLang、NCCL 与 MoE EP": a token sends one payload to each distinct
destination rank among its routes, with a header carrying its route list
(§2.3.2); the destination writes one expert input per route (§2.3.4), runs its
experts, and sends every route's output back into that route's result slot at
the source, which applies the router weight and sums (§3.2, 合对).  Every step of
a rank's data path is a call of the C library (``include/moe.h``: moe_ep_pack,
moe_dispatch_quant_ex, moe_gemm_gateup_down, moe_ep_route_offsets, moe_ep_return,
moe_ep_result_map, moe_combine_packed); the exchanges are the communicator's
all-to-alls (``TorchDistComm``: torch.distributed, NCCL between GPUs).  The
split sizes of an all-to-all are host integers, so each layer call reads the
send counts and the route offsets at the rank boundaries back to the host.

With the tokens of all ranks numbered rank after rank, the slots, capacity
drops and outputs equal those of the one-GPU layer on all the tokens, bit for
bit: rows reach a destination grouped by source rank in ascending token order,
which is ascending global route id.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib
from . import api


class TorchDistComm:
    """All-to-all over a torch.distributed process group."""

    def __init__(self, group=None):
        self.group = group

    def all_to_all(self, out, inp, out_splits, in_splits):
        torch.distributed.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)


class CudaEpOps:
    """The library calls of each phase of a rank's data path."""

    def pack(self, x, topk_idx, E, L):
        lib = _lib.load()
        T, H = x.shape
        K = topk_idx.shape[1]
        W = E // L
        dev = x.device
        rows = max(1, T * min(K, W))
        send_x = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
        send_ids = torch.empty(rows, K, dtype=torch.int32, device=dev)
        send_counts = torch.empty(W, dtype=torch.int32, device=dev)
        route_msg = torch.empty(T, K, dtype=torch.int32, device=dev)
        route_pos = torch.empty(T, K, dtype=torch.int32, device=dev)
        status = torch.empty(2, dtype=torch.int32, device=dev)
        ws = api._workspace(lib.moe_ep_pack_workspace_size(T, K, E, L), dev)
        st = lib.moe_ep_pack(api._p(x), api._p(topk_idx), api._idx_bits(topk_idx), T, H, K, E, L,
                             api._p(send_x), api._p(send_ids), api._p(send_counts), api._p(route_msg),
                             api._p(route_pos), api._p(status), api._p(ws), ws.numel(), api._s(None))
        _lib.check("moe_ep_pack", st)
        return {"send_x": send_x, "send_ids": send_ids, "send_counts": send_counts,
                "route_msg": route_msg, "route_pos": route_pos, "status": status}

    def local(self, recv_x, recv_ids, L, R, weights, gemm_launch=None):
        """The destination's own layer on the received rows, on the fused path:
        dispatch by the rows' local expert ids with the quantisation, then
        both GEMMs."""
        xq, xs, counts, src_map, status = api.moe_dispatch_quant(recv_x, recv_ids, None, L, R)
        out = api.moe_gemm_gateup_down(xq, xs, counts, *weights, dev_status=status,
                                       gemm_launch=gemm_launch)
        return {"out": out, "src_map": src_map, "counts": counts, "status": status}

    def offsets(self, ids):
        lib = _lib.load()
        S, K = ids.shape
        off = torch.empty(S + 1, dtype=torch.int32, device=ids.device)
        ws = api._workspace(lib.moe_ep_offsets_workspace_size(S), ids.device)
        _lib.check("moe_ep_route_offsets",
                   lib.moe_ep_route_offsets(api._p(ids), S, K, api._p(off), api._p(ws), ws.numel(),
                                            api._s(None)))
        return off

    def ret(self, out, src_map, ids, offsets, n_ret):
        lib = _lib.load()
        S, K = ids.shape
        H = out.shape[-1]
        ret_x = torch.empty(max(n_ret, 1), H, dtype=torch.bfloat16, device=out.device)[:n_ret]
        flag = torch.empty(max(n_ret, 1), dtype=torch.int32, device=out.device)[:n_ret]
        st = lib.moe_ep_return(api._p(out), out.numel() // H, api._p(src_map), api._p(ids),
                               api._p(offsets), S, K, H, api._p(ret_x), api._p(flag), api._s(None))
        _lib.check("moe_ep_return", st)
        return ret_x, flag

    def result(self, route_msg, route_pos, offsets, flag, n_ret):
        lib = _lib.load()
        T, K = route_msg.shape
        rm = torch.empty(T, K, dtype=torch.int32, device=route_msg.device)
        st = lib.moe_ep_result_map(api._p(route_msg), api._p(route_pos), api._p(offsets),
                                   api._p(flag), n_ret, T, K, api._p(rm), api._s(None))
        _lib.check("moe_ep_result_map", st)
        return rm

    def combine(self, ret_x, result_map, topk_w, T, H):
        if ret_x.shape[0] == 0:
            ret_x = torch.zeros(1, H, dtype=torch.bfloat16, device=topk_w.device)
        return api.moe_combine_packed(ret_x, result_map, topk_w)


@dataclass
class EpResult:
    y: torch.Tensor            # [T, H] bf16, this rank's tokens
    send_counts: list          # messages sent to each rank (one per token and destination)
    recv_counts: list          # messages received from each rank
    local_counts: torch.Tensor  # [L] rows kept per local expert
    source_status: torch.Tensor  # [2] bad ids of this rank's routes
    local_status: torch.Tensor   # [2] capacity drops at this rank's experts


class ExpertParallelLayer:
    """One rank of an expert-parallel MoE layer: E experts over W = E / L
    ranks, this rank holding experts [rank*L, rank*L + L) with capacity R rows
    each.  ``forward`` takes this rank's tokens and the global router ids and
    returns their routed output; the weights passed are this rank's L experts
    ([L, 2I, H] and [L, H, I] with their block scales)."""

    def __init__(self, E: int, L: int, R: int, rank: int, comm=None, ops=None, gemm_launch=None):
        if E % L:
            raise ValueError("E must be a multiple of L")
        self.E, self.L, self.R, self.W, self.rank = E, L, R, E // L, rank
        self.comm = comm if comm is not None else TorchDistComm()
        self.ops = ops if ops is not None else CudaEpOps()
        self.gemm_launch = gemm_launch

    def forward(self, x, topk_idx, topk_w, w13, w13_scale, w2, w2_scale) -> EpResult:
        ops, comm = self.ops, self.comm
        T, H = x.shape
        K = topk_idx.shape[1]
        dev = x.device
        # source: one payload per (token, destination rank), route lists
        p = ops.pack(x, topk_idx, self.E, self.L)
        recv_counts = torch.empty_like(p["send_counts"])
        comm.all_to_all(recv_counts, p["send_counts"], [1] * self.W, [1] * self.W)
        sc = [int(v) for v in p["send_counts"].tolist()]
        rc = [int(v) for v in recv_counts.tolist()]
        S, Sr = sum(sc), sum(rc)
        recv_x = torch.empty(Sr, H, dtype=torch.bfloat16, device=dev)
        recv_ids = torch.empty(Sr, K, dtype=torch.int32, device=dev)
        comm.all_to_all(recv_x, p["send_x"][:S].contiguous(), rc, sc)
        comm.all_to_all(recv_ids, p["send_ids"][:S].contiguous(), rc, sc)
        # destination: the local experts on the received rows, one returned row per route
        loc = ops.local(recv_x, recv_ids, self.L, self.R, (w13, w13_scale, w2, w2_scale),
                        gemm_launch=self.gemm_launch)
        roff = ops.offsets(recv_ids)
        roff_h = roff.tolist()
        bounds = [0]
        for c in rc:
            bounds.append(bounds[-1] + c)
        ret_send = [roff_h[bounds[s + 1]] - roff_h[bounds[s]] for s in range(self.W)]
        ret_x, flag = ops.ret(loc["out"], loc["src_map"], recv_ids, roff, roff_h[-1])
        # source: the returned rows of its routes, in the order it sent them
        soff = ops.offsets(p["send_ids"][:S])
        soff_h = soff.tolist()
        sb = [0]
        for c in sc:
            sb.append(sb[-1] + c)
        ret_recv = [soff_h[sb[d + 1]] - soff_h[sb[d]] for d in range(self.W)]
        n_back = soff_h[-1]
        back_x = torch.empty(n_back, H, dtype=torch.bfloat16, device=dev)
        back_flag = torch.empty(n_back, dtype=torch.int32, device=dev)
        comm.all_to_all(back_x, ret_x.contiguous(), ret_recv, ret_send)
        comm.all_to_all(back_flag, flag.contiguous(), ret_recv, ret_send)
        result_map = ops.result(p["route_msg"], p["route_pos"], soff, back_flag, n_back)
        y = ops.combine(back_x, result_map, topk_w, T, H)
        return EpResult(y=y, send_counts=sc, recv_counts=rc, local_counts=loc["counts"],
                        source_status=p["status"], local_status=loc["status"])
