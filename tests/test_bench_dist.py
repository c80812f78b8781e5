"""The multi-process path of bench.py on CPU: two gloo ranks (replicas) agree
on the slowest rank's time and the summed work, through the same helpers the
benchmark uses under torchrun."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    r, local, w = bench.dist_setup(world)
    try:
        assert (r, local, w) == (rank, rank, world)
        bench.barrier(w)
        elapsed = 10.0 + 5.0 * r             # rank 1 is the slow one
        rows = 1000.0 * (r + 1)
        mx = bench.reduce_max(elapsed, w, torch.device("cpu"))
        tot = bench.reduce_sum(rows, w, torch.device("cpu"))
        out.put((r, mx, tot))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_max_time_and_summed_rows():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [x[1] for x in res] == [15.0, 15.0]        # max over ranks
    assert [x[2] for x in res] == [3000.0, 3000.0]    # whole-job work


def test_single_process_helpers_are_identity():
    import bench
    assert bench.reduce_max(3.5, 1, None) == 3.5
    assert bench.reduce_sum(2.0, 1, None) == 2.0
    bench.barrier(1)


def test_layer_accounting_matches_formulas():
    """Algorithmic bytes and FLOPs per layer (the roofline numerators)."""
    import bench
    from token_dispatch_grouped_topk_gb300 import workloads as W
    wl = W.WORKLOADS["large"]
    a = bench.layer_bytes_flops(wl, n_valid=131072, n_active_experts=256)
    assert a["gemm_gateup_flops"] == 4 * 131072 * 7168 * 2048
    assert a["gemm_down_flops"] == 2 * 131072 * 7168 * 2048
    assert a["dispatch_bytes"] == 16384 * 7168 * 2 + 16384 * 8 * 8 + 131072 * 7168 * 2 + 16384 * 8 * 4 + 256 * 4
    assert a["combine_bytes"] == 131072 * 7168 * 2 + 2 * 16384 * 8 * 4 + 16384 * 7168 * 2
    assert a["quant_bytes"] == 131072 * (3 * 7168 + 56 * 4)
