"""A reduced, profiler-sized case of the expert-compute kernels.

Runs the per-token FP8 quantisation, the gate/up GEMM (with SiLU*up and the Z
requantisation) and the down GEMM on E experts with `rows` valid rows each and
the large layer's H and I, `reps` times: as two launches, or with --fused as the
one launch the layer uses (down tiles start per 128-row block).  Device memory
stays at a few GB so a full Nsight Compute capture of one launch ends quickly;
inputs still exceed L2.

    python -m token_dispatch_grouped_topk_gb300.profile_case [--E 32] [--rows 512]
           [--H 7168] [--I 2048] [--reps 3] [--fused]

With --dispatch WORKLOAD it instead runs the dispatch fused with the
quantisation (moe_dispatch_quant, padded layout) `reps` times on that named
layer's inputs (seed 0): a capture of the prefill layer holds about 1.1 GB.
"""
import argparse

import torch

from . import api
from . import workloads as W


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--E", type=int, default=32)
    ap.add_argument("--rows", type=int, default=512)
    ap.add_argument("--H", type=int, default=7168)
    ap.add_argument("--I", type=int, default=2048)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--fused", action="store_true")
    ap.add_argument("--dispatch", default=None, choices=["decode", "prefill", "large"])
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    if a.dispatch:
        d = W.make_layer_inputs(a.dispatch, seed=0, device=dev, weights=False)
        wl = d["wl"]
        for _ in range(a.reps):
            _, _, counts, _, st = api.moe_dispatch_quant(d["x"], d["topk_idx"], None, wl.E, wl.R)
        torch.cuda.synchronize()
        print(f"profile case ok: dispatch+quant {a.dispatch} x{a.reps}, kept routes "
              f"{int(counts.sum())}, status {st.cpu().tolist()}")
        return
    E, R, H, I = a.E, a.rows, a.H, a.I
    recv = W.activations(E * R, H, 1, dev).view(E, R, H)
    counts = torch.full((E,), R, dtype=torch.int32, device=dev)
    w13, s13, w2, s2 = W.expert_weights(E, H, I, 2, dev)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    out = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    if a.fused:
        times = {"quant": [], "gemm_gateup_down": []}
        sync = torch.empty(max(256, api._lib.load().moe_gemm_gateup_down_sync_size(E, R, 0)),
                           dtype=torch.uint8, device=dev)
    else:
        times = {"quant": [], "gemm_gateup": [], "gemm_down": []}
    for _ in range(a.reps):
        ev[0].record()
        xq, xs = api.moe_quantize_fp8(recv, counts)
        ev[1].record()
        if a.fused:
            api.moe_gemm_gateup_down(xq, xs, counts, w13, s13, w2, s2, out=out, sync=sync,
                                     dev_status=st)
        else:
            zq, zs = api.moe_gemm_gateup_silu(xq, xs, counts, w13, s13, dev_status=st)
            ev[2].record()
            api.moe_gemm_down(zq, zs, counts, w2, s2, out=out, dev_status=st)
        ev[len(times)].record()
        torch.cuda.synchronize()
        for j, k in enumerate(times):
            times[k].append(ev[j].elapsed_time(ev[j + 1]))
    s = st.cpu().tolist()
    if s != [0, 0]:
        raise SystemExit(f"device status {s}")
    rows = E * R
    best = {k: min(v[1:] or v) for k, v in times.items()}
    rates = {"gemm_gateup": 4.0, "gemm_down": 2.0, "gemm_gateup_down": 6.0}
    print(f"profile case ok: E={E} rows={R} H={H} I={I} reps={a.reps}; best ms "
          + ", ".join(f"{k} {v:.4f}" for k, v in best.items()) + "; "
          + ", ".join(f"{k} {rates[k] * rows * H * I / best[k] / 1e9:.1f} TFLOP/s"
                      for k in best if k in rates))


if __name__ == "__main__":
    main()
