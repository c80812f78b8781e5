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


# The source files each kernel family is compiled from: a recorded ncu figure
# stays valid while these are unchanged.
KERNEL_SOURCES = {
    "gemm": ("gemm.cu", "common.cuh"),
    "dispatch": ("dispatch.cu", "common.cuh"),
    "quant": ("quant.cu", "common.cuh"),
    "combine": ("combine.cu", "common.cuh"),
}


def kernel_sources_digest(kernel: str) -> str:
    family = next((f for f in KERNEL_SOURCES if kernel.startswith(f)), None)
    csrc = os.path.join(ROOT, "token_dispatch_grouped_topk_gb300", "csrc")
    names = KERNEL_SOURCES[family] if family else sorted(os.listdir(csrc))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    item = rec.get(f"{kernel}@{workload}")
    if not item or item.get("sources") != kernel_sources_digest(kernel):
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

def host_description() -> dict:
    """CPU model and core count of this host (the oracle baseline's hardware)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
                             timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"cpu_model": model, "nproc": os.cpu_count()}


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
                       f"combine; plus the full routing pass over {wl.T * wl.K} routes charged pro rata")}


def cpu_oracle_sample_single_thread(wl, n_experts: int, rows_per_expert: int) -> dict | None:
    """The same sample in a child process whose BLAS and OpenMP pools are
    limited to one thread; None if the child fails."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-sample", wl.name,
           "--cpu-experts", str(n_experts), "--cpu-rows", str(rows_per_expert)]
    try:
        p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, env=env,
                           timeout=600)
        return json.loads(p.stdout.strip().splitlines()[-1]) if p.returncode == 0 else None
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def cpu_small_kernels_full(wl, seed: int = 0) -> dict:
    """The oracle's routing, scatter, quantisation and combine over the whole
    batch of a workload (every token, every kept route), timed as they stand;
    the expert MLP is not part of this figure."""
    import oracle as O
    from token_dispatch_grouped_topk_gb300 import workloads as W

    idx, w = W.router(wl.T, wl.E, wl.K, W.router_bias(wl, seed, "cpu"), seed + 1, "cpu")
    x = W.activations(wl.T, wl.H, seed + 2, "cpu").float().numpy()
    idx_np, w_np = idx.numpy(), w.numpy()
    t = {}
    t0 = time.perf_counter()
    rr = O.route(idx_np, wl.E, wl.R)
    t["route"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    recv = O.scatter(x, rr.src_map, wl.E, wl.R).reshape(wl.E * wl.R, wl.H)
    t["scatter"] = time.perf_counter() - t0
    rows = rr.src_map[rr.src_map >= 0]
    t0 = time.perf_counter()
    O.quantize_rows(recv[np.sort(rows)])
    t["quant"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.combine_f32_sequential(recv, rr.src_map, w_np)   # reads only the kept (written) rows
    t["combine"] = time.perf_counter() - t0
    n = int(rr.counts.sum())
    total = sum(t.values())
    return {"rows": n, "seconds": {k: round(v, 4) for k, v in t.items()}, "rows_per_s": n / total,
            "note": f"{wl.name}: T={wl.T} E={wl.E} top-{wl.K} H={wl.H}, every kept route"}


# ------------------------------------------------------------------ GPU arm

def graph_ms(graphs, steps, stream, warmup, world, device, sampler=None, load_s=0.0):
    """Times `steps` CUDA-graph replays (one per routing, cycled) with events
    on the launching stream, barriers and a sync on both sides; returns the
    slowest rank's elapsed ms.  With a clock sampler, `load_s` seconds of the
    same replays run before and after the timed region inside its window."""
    n = len(graphs)
    for i in range(warmup):
        graphs[i % n].replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def load():
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < load_s:
            for i in range(n):
                graphs[i].replay()
            torch.cuda.synchronize()

    def timed():
        barrier(world)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(steps):
            graphs[(warmup + i) % n].replay()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)

    if sampler is None:
        timed()
    else:
        with sampler:
            load()
            timed()
            load()
    return reduce_max(a.elapsed_time(b), world, device)


def capture(fn, n):
    """One CUDA graph per routing r of fn(r)."""
    gs = []
    for r in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(r)
        gs.append(g)
    return gs


def run_ours(args, rank, local, world):
    from token_dispatch_grouped_topk_gb300 import _lib, api
    from token_dispatch_grouped_topk_gb300 import workloads as W

    lib = _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    peaks = load_peaks()
    seed = 1000 * rank
    x = W.activations(wl.T, wl.H, seed + 2, dev)
    w13, s13, w2, s2 = W.expert_weights(wl.E, wl.H, wl.I, seed + 3, dev)
    routings = [W.router(wl.T, wl.E, wl.K, W.router_bias(wl, seed + r, dev), seed + r + 1, dev)
                for r in range(N_ROUTINGS)]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, dev)
    E, R, H, I, K, T = wl.E, wl.R, wl.H, wl.I, wl.K, wl.T
    xq, xs, zq, zs = buf.workspace_views()
    sync = buf.sync_view()
    stream = torch.cuda.current_stream()
    n_gemm = int(lib.moe_expert_compute_gemm_launches(E, R, 0, I, 0))
    form = "one" if n_gemm == 1 else "two"
    rank_offsets = None
    if wl.tokens_per_rank:
        rank_offsets = torch.tensor(np.concatenate([[0], np.cumsum(wl.tokens_per_rank)]),
                                    dtype=torch.int32, device=dev)

    # routing figures of each of the four routings (moe_layer_stats)
    n_valid, n_active, stats = [], [], []
    for idx, w in routings:
        api.moe_dispatch(x, idx, w, E, R, recv=buf.recv, counts=buf.counts, src_map=buf.src_map,
                         dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        st = api.layer_stats_dict(api.moe_layer_stats(idx, buf.counts, wl.L, R, rank_offsets=rank_offsets),
                                  E, R)
        stats.append(st)
        n_valid.append(st["kept_routes"])
        n_active.append(st["active_experts"])

    # One step = the layer as MoeLayerBuffers.forward runs it: dispatch fused
    # with the quantisation (moe_dispatch_quant_ex) -> the GEMMs in the
    # library's launch form for this shape -> combine, with events between
    # the launches (eager loop) for each kernel's time.  The separate path
    # (BF16 dispatch, then quantisation) is timed below as a variant.
    gemm_names = ["gemm_gateup_down"] if form == "one" else ["gemm_gateup", "gemm_down"]

    def layer_step(first, stage_names):
        def step(i, evs=None):
            idx, w = routings[i % N_ROUTINGS]
            rec = (lambda j: evs[j].record(stream)) if evs else (lambda j: None)
            rec(0)
            k = first(x, idx, w, rec)
            if form == "one":
                api.moe_gemm_gateup_down(xq, xs, buf.counts, w13, s13, w2, s2, zq=zq, zs=zs, out=buf.out,
                                         sync=sync, dev_status=buf.dev_status, gemm_launch="one")
            else:
                api.moe_gemm_gateup_silu(xq, xs, buf.counts, w13, s13, zq=zq, zs=zs, dev_status=buf.dev_status)
                k += 1
                rec(k)
                api.moe_gemm_down(zq, zs, buf.counts, w2, s2, out=buf.out, dev_status=buf.dev_status)
            k += 1
            rec(k)
            api.moe_combine(buf.out, buf.src_map, w, y=buf.y)
            rec(k + 1)
        return step

    def fused_first(x_, idx, w, rec):
        api.moe_dispatch_quant(x_, idx, w, E, R, xq=xq, xs=xs, counts=buf.counts, src_map=buf.src_map,
                               dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        rec(1)
        return 1

    def separate_first(x_, idx, w, rec):
        api.moe_dispatch(x_, idx, w, E, R, recv=buf.recv, counts=buf.counts, src_map=buf.src_map,
                         dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        rec(1)
        api.moe_quantize_fp8(buf.recv, buf.counts, xq=xq, xs=xs)
        rec(2)
        return 2

    def time_layer(step, stage_names, sampler=None):
        """Graph-replay ms for args.steps steps, eager ms, per-stage ms."""
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        graphs = capture(step, N_ROUTINGS)
        g_ms = graph_ms(graphs, args.steps, stream, args.warmup, world, dev, sampler=sampler,
                        load_s=0.6 if sampler else 0.0)
        del graphs
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stage_names) + 1)]
               for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0e.record(stream)
        for i in range(args.steps):
            step(args.warmup + i, evs[i])
        t1e.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        if buf.dev_status.cpu().tolist()[0] & api.DEV_TIMEOUT:
            raise RuntimeError("device timeout during the timed region")
        st_ms = {n: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]))
                 for j, n in enumerate(stage_names)}
        return g_ms, t0e.elapsed_time(t1e), st_ms

    stage_names = ["dispatch_quant"] + gemm_names + ["combine"]
    clk = ClockSampler(local)
    elapsed_ms, eager_ms, stage_ms = time_layer(layer_step(fused_first, stage_names), stage_names, sampler=clk)
    sep_names = ["dispatch", "quant"] + gemm_names + ["combine"]
    sep_ms, _, sep_stage_ms = time_layer(layer_step(separate_first, sep_names), sep_names)
    rows_steps = [n_valid[(args.warmup + i) % N_ROUTINGS] for i in range(args.steps)]
    rows_local = float(sum(rows_steps))
    rows_total = reduce_sum(rows_local, world, dev)
    value = rows_total / (elapsed_ms / 1e3)
    mean_rows = rows_total / args.steps / world

    # ---- both launch forms of the GEMMs, same routings, eager with events
    def forms_step(i, fe):
        idx, w = routings[i % N_ROUTINGS]
        api.moe_dispatch_quant(x, idx, w, E, R, xq=xq, xs=xs, counts=buf.counts, src_map=buf.src_map,
                               dev_status=buf.dev_status, workspace=buf.ws_dispatch)
        fe[0].record(stream)
        api.moe_gemm_gateup_down(xq, xs, buf.counts, w13, s13, w2, s2, zq=zq, zs=zs, out=buf.out,
                                 sync=sync, dev_status=buf.dev_status, gemm_launch="one")
        fe[1].record(stream)
        api.moe_gemm_gateup_silu(xq, xs, buf.counts, w13, s13, zq=zq, zs=zs, dev_status=buf.dev_status)
        fe[2].record(stream)
        api.moe_gemm_down(zq, zs, buf.counts, w2, s2, out=buf.out, dev_status=buf.dev_status)
        fe[3].record(stream)

    form_steps = max(3, min(args.steps, 20))
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(form_steps)]
    for i in range(args.warmup):
        forms_step(i, fevs[0])
    torch.cuda.synchronize()
    for i in range(form_steps):
        forms_step(args.warmup + i, fevs[i])
    torch.cuda.synchronize()
    f_ms = {n: float(np.mean([fevs[i][j].elapsed_time(fevs[i][j + 1]) for i in range(form_steps)]))
            for j, n in enumerate(["one_launch", "gate_up", "down"])}
    f_rows = float(np.mean([n_valid[(args.warmup + i) % N_ROUTINGS] for i in range(form_steps)]))

    # ---- packed layout (moe_dispatch_quant_ex / moe_gemm_gateup_down / moe_combine_packed
    # on [rows, ...] buffers), graph replay
    pbuf = api.MoeLayerBuffers(T, E, K, H, I, R, dev, packed=True)
    pgraphs = capture(lambda r: pbuf.forward(x, *routings[r], w13, s13, w2, s2), N_ROUTINGS)
    packed_ms = graph_ms(pgraphs, args.steps, stream, args.warmup, world, dev)

    def lane_bytes(b):
        return int(sum(t.numel() * t.element_size()
                       for t in (b.recv, b.out, b.ws_compute, b.ws_dispatch, b.counts, b.src_map, b.y)))

    packed = {"value": rows_total / (packed_ms / 1e3), "unit": UNIT, "ms_per_step": packed_ms / args.steps,
              "lane_bytes": lane_bytes(pbuf), "padded_lane_bytes": lane_bytes(buf),
              "note": "MoeLayerBuffers(packed=True).forward (moe_dispatch_quant_ex, moe_gemm_gateup_down, "
                      "moe_combine_packed on the packed layout): the receive-side buffers hold "
                      "min(T*K, E*R) rows instead of E*R (CUDA-graph replay); lane bytes count every "
                      "buffer of the lane, the unused BF16 receive buffer included"}
    del pgraphs, pbuf
    torch.cuda.empty_cache()

    # ---- per-source fixed slots (moe_*_source_slots), the decode-path layout:
    # max_tokens = the largest source rank's token count; skipped when its
    # receive buffer would exceed 16 GB
    mt = max(wl.tokens_per_rank) if wl.tokens_per_rank else -(-T // wl.W)
    if wl.W * mt <= R:
        sbuf = api.MoeLayerBuffers(T, E, K, H, I, wl.W * mt, dev, source_slots=mt, L=wl.L,
                                   rank_offsets=rank_offsets)
        sbuf.slots_fp8  # formed outside the capture
        sgraphs = capture(lambda r: sbuf.forward(x, *routings[r], w13, s13, w2, s2), N_ROUTINGS)
        ss_ms = graph_ms(sgraphs, args.steps, stream, args.warmup, world, dev)
        del sgraphs
        sbuf.recv  # the separate path's BF16 slots, formed before its capture
        sgraphs = capture(lambda r: sbuf.forward(x, *routings[r], w13, s13, w2, s2, fused=False),
                          N_ROUTINGS)
        ss_sep_ms = graph_ms(sgraphs, args.steps, stream, args.warmup, world, dev)
        ss_rows = []
        for r in range(N_ROUTINGS):
            sbuf.forward(x, *routings[r], w13, s13, w2, s2)
            ss_rows.append(int(sbuf.counts.sum().item()))
        ss_total = reduce_sum(float(sum(ss_rows[(args.warmup + i) % N_ROUTINGS] for i in range(args.steps))),
                              world, dev)
        common = sum(t.numel() * t.element_size() for t in (sbuf.out, sbuf.ws_compute, sbuf.ws_dispatch,
                                                            sbuf.counts, sbuf.seg_counts, sbuf.src_map,
                                                            sbuf.y))
        source_slots = {"value": ss_total / (ss_ms / 1e3), "unit": UNIT, "ms_per_step": ss_ms / args.steps,
                        "separate_value": ss_total / (ss_sep_ms / 1e3),
                        "separate_ms_per_step": ss_sep_ms / args.steps,
                        "max_tokens": mt, "rows_per_expert": wl.W * mt,
                        "lane_bytes": int(common + sum(t.numel() * t.element_size() for t in sbuf.slots_fp8)),
                        "separate_lane_bytes": int(common + sbuf.recv.numel() * sbuf.recv.element_size()),
                        "note": "MoeLayerBuffers(source_slots).forward: moe_dispatch_quant_source_slots "
                                "(FP8 slots) / moe_gemm_source_slots / moe_combine; separate_*: "
                                "forward(fused=False), moe_dispatch_source_slots (BF16 slots) / "
                                "moe_expert_compute_source_slots / moe_combine. Each source rank owns "
                                "max_tokens slots in every expert (CUDA-graph replay)"}
        del sgraphs, sbuf
        torch.cuda.empty_cache()
    else:
        source_slots = {"skipped": f"W*max_tokens = {wl.W * mt} slot rows per expert exceed the layer's "
                                   f"capacity R = {R}: the layout is the decode path's (every source rank "
                                   f"keeps a full range in every expert)"}

    # ---- two micro-batches: serial split, and overlapped on two streams with
    # the GEMMs' grid capped at several SM counts (the rest left to the other
    # stream's dispatch and combine)
    tbo_steps = max(3, min(args.steps, 20))

    def tbo_ms(overlap, ctas):
        tbo = api.TwoBatchOverlap(T, E, K, H, I, R, dev, gemm_ctas=ctas)
        for i in range(args.warmup):
            tbo.forward(x, *routings[i % N_ROUTINGS], w13, s13, w2, s2, overlap=overlap)
        torch.cuda.synchronize()
        tg = capture(lambda r: tbo.forward(x, *routings[r], w13, s13, w2, s2, overlap=overlap), N_ROUTINGS)
        ms = graph_ms(tg, tbo_steps, stream, args.warmup, world, dev) / tbo_steps
        del tg, tbo
        torch.cuda.empty_cache()
        return ms

    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    tbo_modes = {"no_split": elapsed_ms / args.steps, "serial_split": tbo_ms(False, 0)}
    caps = {}
    for ctas in (0, sm - 8, sm - 24, sm - 40):
        caps[str(ctas or sm)] = tbo_ms(True, ctas)
    tbo_modes["overlapped_split"] = caps[str(sm)]
    best_cap = min(caps, key=caps.get)
    tbo_res = {
        "modes_ms_per_step": tbo_modes,
        "overlapped_by_gemm_ctas_ms": caps, "best_gemm_ctas": int(best_cap),
        "rows_per_s": {k: mean_rows / (v / 1e3) for k, v in tbo_modes.items()},
        "note": "two token halves, one buffer lane each; overlapped = B's dispatch beside A's expert "
                "compute and B's expert compute beside A's combine on two streams; the GEMMs' grid "
                "capped at each listed SM count; every mode timed as CUDA-graph replays",
    }

    # ---- end to end through the public API with host buffers
    x_h = x.cpu().pin_memory()
    r_h = [(i.cpu().pin_memory(), w.cpu().pin_memory()) for i, w in routings]
    y_h = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
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
    # compute of the current one (api.HostPipeline, the layer replayed as one
    # CUDA graph per input slot after the slot's first step); every step still
    # copies its inputs in from pinned host memory and its output back.
    pipe = api.HostPipeline(buf, graph=True)
    y_hs = [y_h, torch.empty_like(y_h).pin_memory()]

    def e2e_step(i):
        ih, wh = r_h[i % N_ROUTINGS]
        pipe.submit(x_h, ih, wh, y_hs[i % 2], w13, s13, w2, s2, stream=stream)

    e2e_steps = max(3, min(args.steps, 20))

    def e2e_time(step_fn, first_stream, last_stream, sampler=None, load_s=0.5):
        for i in range(args.warmup):
            step_fn(i)
        torch.cuda.synchronize()

        def load():
            t0 = time.perf_counter()
            i = 0
            while time.perf_counter() - t0 < load_s:
                step_fn(i)
                i += 1
                if i % 4 == 0:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()

        def timed():
            barrier(world)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(first_stream)
            for i in range(e2e_steps):
                step_fn(args.warmup + i)
            b.record(last_stream)
            torch.cuda.synchronize()
            barrier(world)
            return a.elapsed_time(b)

        if sampler is None:
            ms = timed()
        else:
            with sampler:
                load()
                ms = timed()
                load()
        return reduce_max(ms, world, dev)

    # clocks sampled around the pipelined run (the copies add to the GPU's power draw)
    e2e_clk = ClockSampler(local)
    e2e_ms = e2e_time(e2e_step, pipe.s_in, pipe.s_out, sampler=e2e_clk)
    e2e_serial_ms = e2e_time(e2e_serial_step, stream, stream)
    del pipe
    e2e_rows = reduce_sum(float(sum(n_valid[(args.warmup + i) % N_ROUTINGS] for i in range(e2e_steps))), world, dev)
    h2d = x.numel() * 2 + routings[0][0].numel() * 8 + routings[0][1].numel() * 4
    d2h = T * H * 2

    # ---- the dense FP8 peak of this GPU, measured after every timed region
    # (its seconds of full-power GEMMs would otherwise heat the GPU first)
    fp8 = measure_fp8_peak(dev)

    # ---- rates and the roofline of the dominant kernel
    nv = float(np.mean(rows_steps))
    na = int(round(np.mean([n_active[(args.warmup + i) % N_ROUTINGS] for i in range(args.steps)])))
    acct = layer_bytes_flops(wl, int(nv), na)
    # The kernels are timed inside long loops of layer steps, with the GPU at
    # its power cap, so the FP8 denominator is the sustained cuBLAS rate; the
    # burst rate and the fraction against it are reported beside it.
    fp8_peak = fp8["fp8_tflops_sustained"]
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
    tfs = lambda f, ms: f / (ms * 1e-3) / 1e12
    flops = {"gemm_gateup": acct["gemm_gateup_flops"], "gemm_down": acct["gemm_down_flops"],
             "gemm_gateup_down": acct["gemm_gateup_flops"] + acct["gemm_down_flops"]}
    gbytes = {"gemm_gateup": acct["gemm_gateup_bytes"], "gemm_down": acct["gemm_down_bytes"],
              "gemm_gateup_down": acct["gemm_gateup_bytes"] + acct["gemm_down_bytes"]}
    def kernel_rates(st_ms):
        ks = {}
        for n in st_ms:
            if n in flops:
                ks[n] = {"ms": st_ms[n], "TFLOP/s": tfs(flops[n], st_ms[n]),
                         "frac_fp8": tfs(flops[n], st_ms[n]) / fp8_peak,
                         "GB/s": gbs(gbytes[n], st_ms[n]), "frac_hbm": gbs(gbytes[n], st_ms[n]) / peaks["hbm_gbs"]}
            else:
                b = acct[f"{n}_bytes"]
                ks[n] = {"ms": st_ms[n], "GB/s": gbs(b, st_ms[n]),
                         "frac_hbm": gbs(b, st_ms[n]) / peaks["hbm_gbs"], "bytes": b}
        return ks

    kernels = kernel_rates(stage_ms)
    f_acct = layer_bytes_flops(wl, int(f_rows), na)
    f_fl = f_acct["gemm_gateup_flops"] + f_acct["gemm_down_flops"]
    gemm_forms = {
        "one_launch_ms": f_ms["one_launch"], "two_launches_ms": f_ms["gate_up"] + f_ms["down"],
        "one_launch_TFLOP/s": tfs(f_fl, f_ms["one_launch"]),
        "two_launches_TFLOP/s": tfs(f_fl, f_ms["gate_up"] + f_ms["down"]),
        "gate_up_TFLOP/s": tfs(f_acct["gemm_gateup_flops"], f_ms["gate_up"]),
        "down_TFLOP/s": tfs(f_acct["gemm_down_flops"], f_ms["down"]),
        "chosen": form, "steps": form_steps,
        "note": "both GEMMs in one launch (moe_gemm_gateup_down, tile events) against the gate/up "
                "launch then the down launch, on the same routings; moe_expert_compute picks by "
                "tile count (one launch when the gate/up tiles fill at most 16 waves of SMs)",
    }
    dom = max(stage_names, key=lambda n: stage_ms[n])
    if dom in flops:
        t_tensor = flops[dom] / (fp8_peak * 1e12)
        t_hbm = gbytes[dom] / (peaks["hbm_gbs"] * 1e9)
        if t_tensor >= t_hbm:
            ach = kernels[dom]["TFLOP/s"]
            roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": ach / fp8_peak, "frac_of_burst": ach / fp8["fp8_tflops"],
                    "peak_note": (f"of measured: dense e4m3 cuBLASLt GEMM on this GPU run back to back "
                                  f"for 4 s (sustained {fp8['fp8_tflops_sustained']:.0f} TFLOP/s, the "
                                  f"figure for a kernel timed inside a long loop of steps); its best "
                                  f"single call (burst) {fp8['fp8_tflops']:.0f}; 2 x the measured bf16 "
                                  f"burst would be {2 * peaks['bf16_tflops']:.0f}")}
        else:
            ach = kernels[dom]["GB/s"]
            roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / peaks["hbm_gbs"],
                    "peak_note": (f"of {peaks['source']} HBM copy bandwidth; tensor frac "
                                  f"{kernels[dom]['frac_fp8']:.3f} of the measured sustained fp8 rate "
                                  f"{fp8_peak:.0f}")}
        roof["roofline_ms"] = {"tensor": t_tensor * 1e3, "hbm": t_hbm * 1e3}
        roof["algorithmic"] = {"flops_per_launch": flops[dom], "bytes_per_launch": gbytes[dom]}
    else:
        ach = kernels[dom]["GB/s"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_note": f"of {peaks['source']} HBM copy bandwidth",
                "algorithmic": {"bytes_per_launch": acct[f"{dom}_bytes"]}}
    roof["traffic"] = recorded_traffic(dom, wl.name)
    separate = {
        "value": rows_total / (sep_ms / 1e3), "unit": UNIT, "ms_per_step": sep_ms / args.steps,
        "note": "MoeLayerBuffers.forward(fused=False): moe_dispatch (BF16 rows into the receive buffer), "
                "then the quantisation kernel, the same GEMMs and combine (CUDA-graph replay; per-kernel "
                "times from an eager loop)",
        "kernels": kernel_rates(sep_stage_ms),
    }
    dispatch_kernels = 1 if T * K <= 4096 else 3
    launches_per_step = dispatch_kernels + n_gemm + 1
    return {
        "value": value, "ms_per_step": elapsed_ms / args.steps, "eager_ms_per_step": eager_ms / args.steps,
        "kernels": kernels, "gemm_forms": gemm_forms, "roofline": roof,
        "peaks": {"fp8": fp8, "hbm_copy_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                  "source": peaks["source"]},
        "e2e": {"value": e2e_rows / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
                "path": "api.HostPipeline(graph=True): pinned host in/out every step; step i+1's "
                        "copy-in and step i-1's copy-out run on two copy streams beside step i's "
                        "compute, a CUDA-graph replay of the layer",
                "clocks": e2e_clk.summary(),
                "serial_value": e2e_rows / (e2e_serial_ms / 1e3),
                "serial_note": "copy in, compute, copy out back to back on one stream"},
        "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
        "clocks": clk.summary(), "separate": separate, "tbo": tbo_res, "packed": packed,
        "source_slots": source_slots, "layer_stats": stats,
        "rows_per_step": nv, "wl": wl,
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


def cpu_baseline(wl) -> dict:
    """The oracle as it stands on this host: the bounded expert sample with
    all threads and with one, plus the routing/scatter/quant/combine passes in
    full on the decode- and prefill-shaped layers."""
    from token_dispatch_grouped_topk_gb300 import workloads as W
    host = host_description()
    allt = cpu_oracle_sample(wl, n_experts=8, rows_per_expert=128)
    one = cpu_oracle_sample_single_thread(wl, n_experts=8, rows_per_expert=128)
    small = {n: cpu_small_kernels_full(W.WORKLOADS[n]) for n in ("decode", "prefill")}
    return {"value": allt["value"], "unit": UNIT, "cores": host["nproc"], "threads": host["nproc"],
            "cpu_model": host["cpu_model"], "kind": "oracle", "sample": allt["sample"],
            "single_thread": None if one is None else {"value": one["value"], "unit": UNIT, "threads": 1},
            "routing_scatter_quant_combine_full": small,
            "note": "numpy's BLAS pool takes every core (threads); the single-thread figure runs the "
                    "same sample in a child process with the BLAS/OpenMP pools at one thread"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large", choices=["large", "prefill", "decode", "traced"])
    # internal: one oracle sample as a JSON line (the single-thread baseline's child process)
    ap.add_argument("--cpu-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-experts", type=int, default=8, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-rows", type=int, default=128, help=argparse.SUPPRESS)
    args = ap.parse_args()
    from token_dispatch_grouped_topk_gb300 import workloads as W
    if args.cpu_sample:
        print(json.dumps(cpu_oracle_sample(W.WORKLOADS[args.cpu_sample], args.cpu_experts, args.cpu_rows)))
        return
    if args.warmup < 3:
        args.warmup = 3
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
                                           "path": "MoeLayerBuffers.forward: moe_dispatch_quant_ex -> "
                                                   "grouped GEMMs -> moe_combine",
                                           "eager_ms_per_step": res["eager_ms_per_step"],
                                           "launches_per_step": res["launches_per_step"]}),
            "kernels": res["kernels"], "gemm_forms": res["gemm_forms"], "roofline": res["roofline"],
            "peaks": res["peaks"], "e2e": res["e2e"], "gpu_launches": res["gpu_launches"],
            "clocks": res["clocks"], "layer_stats": res["layer_stats"],
            "separate_dispatch_quant": res["separate"], "packed_layout": res["packed"],
            "source_slots_layout": res["source_slots"], "two_batch_overlap": res["tbo"],
        }
        # the oracle's CPU baseline: rank 0 of a one-GPU run only
        line["cpu_baseline"] = cpu_baseline(wl) if world == 1 else None
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
    host = host_description()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(wl),
        "cpu_baseline": {"kind": "oracle", "cores": host["nproc"], "cpu_model": host["cpu_model"],
                         "sample": vals[0]["sample"], "value": value, "unit": UNIT},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
