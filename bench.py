"""Benchmark of the routed MoE branch on GB300: dispatch -> FP8 quant -> grouped
gated-SiLU FP8 expert MLP -> weighted combine, one step = one layer pass over
one batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload large|prefill|decode|traced]

Prints one JSON line (rank 0).  Default workload: the large layer (T=16384
tokens, E=256 experts as 32 logical ranks x 8, top-8, H=7168, I=2048, R=4096).
Inputs are resident in HBM and larger than L2; the router output changes every
step (four seeded routings, cycled).  Under torchrun (N > 1) every rank runs an
independent replica of the layer on its own GPU (the path has no exchange step
on one GPU), the timed region is bracketed by barriers and the slowest rank's
time is used.

``--impl reference`` times the CPU oracle (``oracle/``) on a bounded sample of
the same workload on the host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "routed token-rows/s per MoE layer"
UNIT = "rows/s"
N_ROUTINGS = 4


# ------------------------------------------------------------------ accounting

def layer_bytes_flops(wl, n_valid: int, n_active_experts: int) -> dict:
    """Algorithmic bytes / FLOPs per layer (what the method must move)."""
    T, K, H, I, E = wl.T, wl.K, wl.H, wl.I, wl.E
    G, GI = H // 128, I // 128
    w13 = n_active_experts * (2 * I * H + (2 * I // 128) * G * 4)
    w2 = n_active_experts * (H * I + G * GI * 4)
    return {
        "dispatch_bytes": T * H * 2 + T * K * 8 + n_valid * H * 2 + T * K * 4 + E * 4,
        "quant_bytes": n_valid * (2 * H + H + G * 4),
        "dispatch_quant_bytes": T * H * 2 + T * K * 8 + n_valid * (H + G * 4) + T * K * 4 + E * 4,
        "gemm_gateup_bytes": w13 + n_valid * (H + G * 4) + n_valid * (I + GI * 4),
        "gemm_down_bytes": w2 + n_valid * (I + GI * 4) + n_valid * H * 2,
        "combine_bytes": n_valid * H * 2 + 2 * T * K * 4 + T * H * 2,
        "gemm_gateup_flops": 4 * n_valid * H * I,
        "gemm_down_flops": 2 * n_valid * H * I,
    }


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def measure_fp8_peak(device, n: int = 8192, sustained_s: float = 4.0) -> dict:
    """Dense e4m3 GEMM throughput of this GPU through cuBLASLt
    (torch._scaled_mm, per-tensor scales, BF16 output), n^3 with 2 n^3 FLOPs:
    the best of 10 timed calls (burst) and the rate of calls back to back for
    `sustained_s` seconds (sustained, under the power cap)."""
    g = torch.Generator(device=device)
    g.manual_seed(0)
    a = torch.randn(n, n, device=device, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=device, generator=g).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device=device, dtype=torch.float32)
    mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    flops = 2.0 * n ** 3
    best = float("inf")
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        mm()
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e))
    # sustained: batches of 20 calls until sustained_s has passed
    calls, t0 = 0, time.perf_counter()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    while time.perf_counter() - t0 < sustained_s:
        for _ in range(20):
            mm()
        calls += 20
        torch.cuda.synchronize()
    e.record()
    e.synchronize()
    sus_ms = s.elapsed_time(e) / calls
    del a, b
    torch.cuda.empty_cache()
    return {"fp8_tflops": flops / (best * 1e-3) / 1e12, "fp8_tflops_sustained": flops / (sus_ms * 1e-3) / 1e12,
            "how": f"torch._scaled_mm e4m3 {n}^3 (2n^3 FLOPs), per-tensor scales, bf16 out: best of 10 "
                   f"(burst) and {calls} calls back to back over {sustained_s:.0f} s (sustained)"}


def kernel_sources_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "token_dispatch_grouped_topk_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    item = rec.get(f"{kernel}@{workload}")
    if not item or item.get("sources") != kernel_sources_digest():
        return None
    return item.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    return rank, local, world


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


# ------------------------------------------------------------------ CPU oracle

def cpu_oracle_sample(wl, n_experts: int, rows_per_expert: int, seed: int = 0) -> dict:
    """Times the oracle, as it stands, on a bounded sample of the workload:
    the routing pass over the whole batch (charged pro rata to the sampled
    rows) and, for `rows_per_expert` kept routes on each of `n_experts`
    experts, quantisation, gate/up GEMM, SiLU*up, requant, down GEMM and the
    weighted combine.  Returns rows/s over the sample."""
    import oracle as O
    from token_dispatch_grouped_topk_gb300 import workloads as W

    idx, w = W.router(wl.T, wl.E, wl.K, W.router_bias(wl, seed, "cpu"), seed + 1, "cpu")
    idx_np, w_np = idx.numpy(), w.numpy()
    t0 = time.perf_counter()
    rr = O.route(idx_np, wl.E, wl.R)
    t_route = time.perf_counter() - t0
    n_valid = int(rr.counts.sum())
    experts = list(np.argsort(-rr.counts)[:n_experts])
    x = W.activations(n_experts * rows_per_expert, wl.H, seed + 2, "cpu").float().numpy()
    w13, s13, w2, s2 = W.expert_weights(n_experts, wl.H, wl.I, seed + 3, "cpu")
    t1 = time.perf_counter()
    rows = 0
    for j, e in enumerate(experts):
        xs = x[j * rows_per_expert:(j + 1) * rows_per_expert]
        xq, sx = O.quantize_rows(xs)
        out, _, _, _ = O.expert_forward(xq, sx, w13[j].numpy(), s13[j].numpy(), w2[j].numpy(), s2[j].numpy())
        sm = np.arange(len(xs), dtype=np.int32)[:, None]
        O.combine_fp64(out, sm, np.ones((len(xs), 1), np.float32))
        rows += len(xs)
    t_exp = time.perf_counter() - t1
    total = t_route * rows / max(n_valid, 1) + t_exp
    return {"value": rows / total, "unit": UNIT, "seconds": t_route + t_exp, "rows": rows,
            "sample": (f"{rows} kept routes of the {wl.name} layer on its {n_experts} busiest experts "
                       f"({rows_per_expert} rows each): quant, gate/up GEMM, SiLU*up, requant, down GEMM, "
                       f"combine; plus the full routing pass over {wl.T * wl.K} routes charged pro rata"),
            "cores": int(torch.get_num_threads())}


# ------------------------------------------------------------------ GPU arm

def run_ours(args, rank, local, world):
    from token_dispatch_grouped_topk_gb300 import _lib, api
    from token_dispatch_grouped_topk_gb300 import workloads as W

    _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    seed = 1000 * rank
    x = W.activations(wl.T, wl.H, seed + 2, dev)
    w13, s13, w2, s2 = W.expert_weights(wl.E, wl.H, wl.I, seed + 3, dev)
    routings = [W.router(wl.T, wl.E, wl.K, W.router_bias(wl, seed + r, dev), seed + r + 1, dev)
                for r in range(N_ROUTINGS)]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    E, R, H, I = wl.E, wl.R, wl.H, wl.I
    xq, xs, zq, zs = buf.workspace_views()
    stream = torch.cuda.current_stream()

    n_valid, n_active = [], []
    for idx, w in routings:
        api.moe_dispatch(x, idx, w, E, R, recv=buf.recv, counts=buf.counts, src_map=buf.src_map,
                         dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        c = buf.counts.cpu()
        n_valid.append(int(c.sum()))
        n_active.append(int((c > 0).sum()))
    dropped = int(buf.dev_status[1].item())

    # One step = dispatch -> quantisation -> both GEMMs in one launch ->
    # combine (the kernels moe_dispatch, moe_expert_compute and moe_combine
    # run), each stage bracketed by events on the launching stream so every
    # launch's duration is measured in place.
    stage_names = ["dispatch", "quant", "gemm_gateup_down", "combine"]
    n_stage = len(stage_names)
    sync = buf.sync_view()

    def step(i, evs=None):
        idx, w = routings[i % N_ROUTINGS]
        if evs: evs[0].record(stream)
        api.moe_dispatch(x, idx, w, E, R, recv=buf.recv, counts=buf.counts, src_map=buf.src_map,
                         dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        if evs: evs[1].record(stream)
        api.moe_quantize_fp8(buf.recv, buf.counts, xq=xq, xs=xs)
        if evs: evs[2].record(stream)
        api.moe_gemm_gateup_down(xq, xs, buf.counts, w13, s13, w2, s2, zq=zq, zs=zs, out=buf.out,
                                 sync=sync, dev_status=buf.dev_status)
        if evs: evs[3].record(stream)
        api.moe_combine(buf.out, buf.src_map, w, y=buf.y)
        if evs: evs[4].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # The headline timing replays one captured CUDA graph per routing (the
    # layer's launches recorded once; the device work is identical).
    graphs = []
    for r in range(N_ROUTINGS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(r)
        graphs.append(g)
    for i in range(args.warmup):
        graphs[i % N_ROUTINGS].replay()
    torch.cuda.synchronize()
    gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        gs.record(stream)
        for i in range(args.steps):
            graphs[(args.warmup + i) % N_ROUTINGS].replay()
        ge.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = gs.elapsed_time(ge)
    del graphs
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_stage + 1)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step(args.warmup + i, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    eager_ms = start.elapsed_time(end)

    status = buf.dev_status.cpu().tolist()
    if status[0] & api.DEV_TIMEOUT:
        raise RuntimeError("device timeout during the timed region")
    stage_ms = {n: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]))
                for j, n in enumerate(stage_names)}

    # ---- the two GEMMs as separate launches (moe_gemm_gateup_silu, then
    # moe_gemm_down), for the rate of each GEMM on its own
    def split_step(i, se):
        idx, w = routings[i % N_ROUTINGS]
        api.moe_dispatch(x, idx, w, E, R, recv=buf.recv, counts=buf.counts, src_map=buf.src_map,
                         dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        api.moe_quantize_fp8(buf.recv, buf.counts, xq=xq, xs=xs)
        se[0].record(stream)
        api.moe_gemm_gateup_silu(xq, xs, buf.counts, w13, s13, zq=zq, zs=zs, dev_status=buf.dev_status)
        se[1].record(stream)
        api.moe_gemm_down(zq, zs, buf.counts, w2, s2, out=buf.out, dev_status=buf.dev_status)
        se[2].record(stream)
        api.moe_combine(buf.out, buf.src_map, w, y=buf.y)

    split_steps = max(3, min(args.steps, 30))
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(split_steps)]
    for i in range(args.warmup):
        split_step(i, sevs[0])
    torch.cuda.synchronize()
    for i in range(split_steps):
        split_step(args.warmup + i, sevs[i])
    torch.cuda.synchronize()
    split_ms = {n: float(np.mean([sevs[i][j].elapsed_time(sevs[i][j + 1]) for i in range(split_steps)]))
                for j, n in enumerate(["gemm_gateup", "gemm_down"])}
    split_rows = float(np.mean([n_valid[(args.warmup + i) % N_ROUTINGS] for i in range(split_steps)]))

    # ---- the same layer with dispatch and quantisation fused (moe_dispatch_quant)
    fused_names = ["dispatch_quant", "gemm_gateup_down", "combine"]

    def fused_step(i, fe=None):
        idx, w = routings[i % N_ROUTINGS]
        if fe: fe[0].record(stream)
        api.moe_dispatch_quant(x, idx, w, E, R, xq=xq, xs=xs, counts=buf.counts, src_map=buf.src_map,
                               dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        if fe: fe[1].record(stream)
        api.moe_gemm_gateup_down(xq, xs, buf.counts, w13, s13, w2, s2, zq=zq, zs=zs, out=buf.out,
                                 sync=sync, dev_status=buf.dev_status)
        if fe: fe[2].record(stream)
        api.moe_combine(buf.out, buf.src_map, w, y=buf.y)
        if fe: fe[3].record(stream)

    for i in range(args.warmup):
        fused_step(i)
    torch.cuda.synchronize()
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fused_names) + 1)]
            for _ in range(args.steps)]
    fs, fe_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    fs.record(stream)
    for i in range(args.steps):
        fused_step(args.warmup + i, fevs[i])
    fe_.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    fused_eager_ms = fs.elapsed_time(fe_)
    fgraphs = []
    for r in range(N_ROUTINGS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fused_step(r)
        fgraphs.append(g)
    for i in range(args.warmup):
        fgraphs[i % N_ROUTINGS].replay()
    torch.cuda.synchronize()
    barrier(world)
    fs.record(stream)
    for i in range(args.steps):
        fgraphs[(args.warmup + i) % N_ROUTINGS].replay()
    fe_.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    fused_ms = reduce_max(fs.elapsed_time(fe_), world, dev)
    del fgraphs
    fused_stage_ms = {n: float(np.mean([fevs[i][j].elapsed_time(fevs[i][j + 1]) for i in range(args.steps)]))
                      for j, n in enumerate(fused_names)}
    rows_steps = [n_valid[(args.warmup + i) % N_ROUTINGS] for i in range(args.steps)]
    rows_local = float(sum(rows_steps))
    max_ms = reduce_max(elapsed_ms, world, dev)
    rows_total = reduce_sum(rows_local, world, dev)
    value = rows_total / (max_ms / 1e3)

    # ---- packed layout (moe_*_packed): the same step with the experts' rows
    # back to back instead of one capacity block per expert
    pbuf = api.MoeLayerBuffers(wl.T, E, wl.K, H, I, R, dev, packed=True)

    def packed_step(i):
        idx, w = routings[i % N_ROUTINGS]
        pbuf.forward(x, idx, w, w13, s13, w2, s2)

    for i in range(args.warmup):
        packed_step(i)
    torch.cuda.synchronize()
    pgraphs = []
    for r in range(N_ROUTINGS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            packed_step(r)
        pgraphs.append(g)
    for i in range(args.warmup):
        pgraphs[i % N_ROUTINGS].replay()
    torch.cuda.synchronize()
    barrier(world)
    fs.record(stream)
    for i in range(args.steps):
        pgraphs[(args.warmup + i) % N_ROUTINGS].replay()
    fe_.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    packed_ms = reduce_max(fs.elapsed_time(fe_), world, dev)

    def lane_bytes(b):
        return int(sum(t.numel() * t.element_size()
                       for t in (b.recv, b.out, b.ws_compute, b.ws_dispatch, b.counts, b.src_map, b.y)))

    packed = {"value": rows_total / (packed_ms / 1e3), "unit": UNIT, "ms_per_step": packed_ms / args.steps,
              "lane_bytes": lane_bytes(pbuf), "padded_lane_bytes": lane_bytes(buf),
              "note": "moe_dispatch_packed / moe_expert_compute_packed / moe_combine_packed: the "
                      "receive-side buffers hold min(T*K, E*R) rows instead of E*R (CUDA-graph replay)"}
    del pgraphs, pbuf
    torch.cuda.empty_cache()

    # ---- two micro-batches: serial split and overlapped on two streams
    tbo = api.TwoBatchOverlap(wl.T, E, wl.K, H, I, R, dev)
    tbo_steps = max(3, min(args.steps, 20))

    def tbo_ms(overlap):
        # one CUDA graph per routing holds the whole split step (both lanes and,
        # when overlapped, both side streams forked from the capturing stream)
        for i in range(args.warmup):
            idx, w = routings[i % N_ROUTINGS]
            tbo.forward(x, idx, w, w13, s13, w2, s2, overlap=overlap)
        torch.cuda.synchronize()
        tgraphs = []
        for r in range(N_ROUTINGS):
            idx, w = routings[r]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                tbo.forward(x, idx, w, w13, s13, w2, s2, overlap=overlap)
            tgraphs.append(g)
        for i in range(args.warmup):
            tgraphs[i % N_ROUTINGS].replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(tbo_steps):
            tgraphs[(args.warmup + i) % N_ROUTINGS].replay()
        b.record(stream)
        torch.cuda.synchronize()
        del tgraphs
        return a.elapsed_time(b) / tbo_steps

    split_serial_ms = tbo_ms(False)
    split_overlap_ms = tbo_ms(True)
    del tbo
    torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers
    x_h = x.cpu().pin_memory()
    r_h = [(i.cpu().pin_memory(), w.cpu().pin_memory()) for i, w in routings]
    y_h = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)
    idx_d = torch.empty_like(routings[0][0])
    w_d = torch.empty_like(routings[0][1])

    def e2e_serial_step(i):
        ih, wh = r_h[i % N_ROUTINGS]
        x_d.copy_(x_h, non_blocking=True)
        idx_d.copy_(ih, non_blocking=True)
        w_d.copy_(wh, non_blocking=True)
        y = buf.forward(x_d, idx_d, w_d, w13, s13, w2, s2)
        y_h.copy_(y, non_blocking=True)

    # The public host-memory path: copies of neighbouring steps overlap the
    # compute of the current one (api.HostPipeline); every step still copies
    # its inputs in from pinned host memory and its output back.
    pipe = api.HostPipeline(buf)
    y_hs = [y_h, torch.empty_like(y_h).pin_memory()]

    def e2e_step(i):
        ih, wh = r_h[i % N_ROUTINGS]
        pipe.submit(x_h, ih, wh, y_hs[i % 2], w13, s13, w2, s2, stream=stream)

    e2e_steps = max(3, min(args.steps, 20))

    def e2e_time(step_fn, first_stream, last_stream):
        for i in range(args.warmup):
            step_fn(i)
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(first_stream)
        for i in range(e2e_steps):
            step_fn(args.warmup + i)
        b.record(last_stream)
        torch.cuda.synchronize()
        barrier(world)
        return reduce_max(a.elapsed_time(b), world, dev)

    e2e_ms = e2e_time(e2e_step, pipe.s_in, pipe.s_out)
    e2e_serial_ms = e2e_time(e2e_serial_step, stream, stream)
    del pipe
    e2e_rows = reduce_sum(float(sum(n_valid[(args.warmup + i) % N_ROUTINGS] for i in range(e2e_steps))), world, dev)
    h2d = x.numel() * 2 + routings[0][0].numel() * 8 + routings[0][1].numel() * 4
    d2h = wl.T * wl.H * 2

    # ---- roofline of the dominant kernel (the two-GEMM launch) and per-kernel rates
    peaks = load_peaks()
    nv = float(np.mean(rows_steps))
    na = int(round(np.mean([n_active[(args.warmup + i) % N_ROUTINGS] for i in range(args.steps)])))

    acct = layer_bytes_flops(wl, int(nv), na)
    fp8_peak = 2.0 * peaks["bf16_tflops"]        # nominal fp8 : bf16 dense ratio 4.5 / 2.25
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
    tfs = lambda f, ms: f / (ms * 1e-3) / 1e12
    gemm_flops = acct["gemm_gateup_flops"] + acct["gemm_down_flops"]
    gemm_bytes = acct["gemm_gateup_bytes"] + acct["gemm_down_bytes"]
    g12 = tfs(gemm_flops, stage_ms["gemm_gateup_down"])
    # the separate-launch GEMM rates, on the rows of the steps they ran
    sacct = layer_bytes_flops(wl, int(split_rows), na)
    g1 = tfs(sacct["gemm_gateup_flops"], split_ms["gemm_gateup"])
    g2 = tfs(sacct["gemm_down_flops"], split_ms["gemm_down"])
    kernels = {
        "dispatch": {"ms": stage_ms["dispatch"], "GB/s": gbs(acct["dispatch_bytes"], stage_ms["dispatch"]),
                     "frac_hbm": gbs(acct["dispatch_bytes"], stage_ms["dispatch"]) / peaks["hbm_gbs"]},
        "quant": {"ms": stage_ms["quant"], "GB/s": gbs(acct["quant_bytes"], stage_ms["quant"]),
                  "frac_hbm": gbs(acct["quant_bytes"], stage_ms["quant"]) / peaks["hbm_gbs"]},
        "gemm_gateup_down": {"ms": stage_ms["gemm_gateup_down"], "TFLOP/s": g12, "frac_fp8": g12 / fp8_peak,
                             "GB/s": gbs(gemm_bytes, stage_ms["gemm_gateup_down"]),
                             "note": "both GEMMs in one launch (moe_gemm_gateup_down)"},
        "combine": {"ms": stage_ms["combine"], "GB/s": gbs(acct["combine_bytes"], stage_ms["combine"]),
                    "frac_hbm": gbs(acct["combine_bytes"], stage_ms["combine"]) / peaks["hbm_gbs"]},
        "separate_launches": {
            "gemm_gateup": {"ms": split_ms["gemm_gateup"], "TFLOP/s": g1, "frac_fp8": g1 / fp8_peak,
                            "GB/s": gbs(sacct["gemm_gateup_bytes"], split_ms["gemm_gateup"])},
            "gemm_down": {"ms": split_ms["gemm_down"], "TFLOP/s": g2, "frac_fp8": g2 / fp8_peak,
                          "GB/s": gbs(sacct["gemm_down_bytes"], split_ms["gemm_down"])},
            "steps": split_steps,
            "note": "moe_gemm_gateup_silu then moe_gemm_down (eager, events around each)"},
    }
    mean_rows = rows_total / args.steps / world
    tbo_res = {
        "modes_ms_per_step": {"no_split": max_ms / args.steps, "serial_split": split_serial_ms,
                              "overlapped_split": split_overlap_ms},
        "rows_per_s": {"no_split": value, "serial_split": mean_rows / (split_serial_ms / 1e3),
                       "overlapped_split": mean_rows / (split_overlap_ms / 1e3)},
        "note": "two token halves, one buffer lane each; overlapped = B's dispatch beside A's expert "
                "compute and B's expert compute beside A's combine on two streams; every mode "
                "timed as CUDA-graph replays",
    }
    fused = {
        "value": rows_total / (fused_ms / 1e3), "unit": UNIT, "ms_per_step": fused_ms / args.steps,
        "note": "moe_dispatch_quant (each token row quantised once, FP8 scattered) replaces dispatch + quant",
        "kernels": {
            "dispatch_quant": {"ms": fused_stage_ms["dispatch_quant"],
                               "GB/s": gbs(acct["dispatch_quant_bytes"], fused_stage_ms["dispatch_quant"]),
                               "frac_hbm": gbs(acct["dispatch_quant_bytes"], fused_stage_ms["dispatch_quant"]) / peaks["hbm_gbs"]},
            "gemm_gateup_down": {"ms": fused_stage_ms["gemm_gateup_down"]},
            "combine": {"ms": fused_stage_ms["combine"]},
        },
        "gpu_launches": 5 * args.steps,
    }
    dom = max(stage_ms, key=stage_ms.get)
    if dom == "gemm_gateup_down":
        # The GEMM launch's bound is whichever roofline time is longer: its
        # FLOPs at the FP8 peak or its bytes at the HBM peak (decode-shaped
        # layers stream the weights for few rows and sit below the ridge).
        t_tensor = gemm_flops / (fp8_peak * 1e12)
        t_hbm = gemm_bytes / (peaks["hbm_gbs"] * 1e9)
        if t_tensor >= t_hbm:
            achieved = kernels[dom]["TFLOP/s"]
            roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                    "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                    "peak_note": f"fp8 dense = 2 x bf16 burst of {peaks['source']} peaks"}
        else:
            achieved = kernels[dom]["GB/s"]
            roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_note": f"{peaks['source']} HBM copy bandwidth; tensor frac "
                                 f"{kernels[dom]['frac_fp8']:.3f} of the fp8 dense peak"}
        roof["roofline_ms"] = {"tensor": t_tensor * 1e3, "hbm": t_hbm * 1e3}
        roof["traffic"] = recorded_traffic(dom, wl.name)
    else:
        achieved = kernels[dom]["GB/s"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_note": f"{peaks['source']} HBM copy bandwidth",
                "traffic": recorded_traffic(dom, wl.name)}
    return {
        "value": value, "ms_per_step": max_ms / args.steps, "eager_ms_per_step": eager_ms / args.steps,
        "kernels": kernels, "roofline": roof,
        "e2e": {"value": e2e_rows / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
                "path": "api.HostPipeline: pinned host in/out every step; step i+1's copy-in and "
                        "step i-1's copy-out run on two copy streams beside step i's compute",
                "serial_value": e2e_rows / (e2e_serial_ms / 1e3),
                "serial_note": "copy in, compute, copy out back to back on one stream"},
        "gpu_launches": 6 * args.steps, "clocks": clk.summary(), "fused": fused, "tbo": tbo_res,
        "packed": packed,
        "rows_per_step": nv, "dropped_routes_last_routing": dropped, "wl": wl,
    }


def workload_config(wl, extra=None) -> dict:
    x_mb = wl.T * wl.H * 2 / 1e6
    w_gb = wl.E * 3 * wl.H * wl.I / 1e9
    if x_mb > 129:
        l2 = (f"inputs larger than L2 (no flush): x ({x_mb:.0f} MB) and the FP8 weights "
              f"({w_gb:.1f} GB) exceed 129 MB")
    else:
        l2 = (f"no separate flush: every step streams the FP8 weights ({w_gb:.1f} GB, larger "
              f"than the 129 MB L2) between two uses of x ({x_mb:.1f} MB), which evicts it")
    cfg = {"workload": f"{wl.name}: T={wl.T} E={wl.E} ({wl.W}x{wl.L}) top-{wl.K} H={wl.H} I={wl.I} R={wl.R}",
           "global_batch": wl.T, "routings": N_ROUTINGS, "l2": l2}
    if extra:
        cfg.update(extra)
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large", choices=["large", "prefill", "decode", "traced"])
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from token_dispatch_grouped_topk_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]

    rank, local, world = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl, world)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    res = run_ours(args, rank, local, world)
    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded; random-init block-FP8 weights)",
            "config": workload_config(wl, {"parallelism": f"replicas x{world}",
                                           "rows_per_step": res["rows_per_step"],
                                           "timing": "CUDA-graph replay of each step (per-kernel "
                                                     "times from an eager loop with events)",
                                           "eager_ms_per_step": res["eager_ms_per_step"]}),
            "kernels": res["kernels"], "roofline": res["roofline"], "e2e": res["e2e"],
            "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
            "fused_dispatch_quant": res["fused"],
            "packed_layout": res["packed"],
            "two_batch_overlap": res["tbo"],
        }
        sample = cpu_oracle_sample(wl, n_experts=8, rows_per_expert=128)
        line["cpu_baseline"] = {"value": sample["value"], "unit": UNIT, "cores": sample["cores"],
                                "kind": "oracle", "sample": sample["sample"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, wl, world):
    """The CPU oracle as the reference arm: each step one bounded sample."""
    vals = []
    for i in range(args.warmup + args.steps):
        s = cpu_oracle_sample(wl, n_experts=1, rows_per_expert=32, seed=i)
        if i >= args.warmup:
            vals.append(s)
    secs = sum(v["seconds"] for v in vals)
    value = float(np.mean([v["value"] for v in vals]))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(wl),
        "cpu_baseline": {"kind": "oracle", "cores": vals[0]["cores"], "sample": vals[0]["sample"], "value": value,
                         "unit": UNIT},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
