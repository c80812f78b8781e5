"""A reduced, profiler-sized case of the expert-compute kernels.

Runs the per-token FP8 quantisation, the gate/up GEMM (with SiLU*up and the Z
requantisation) and the down GEMM on E experts with `rows` valid rows each and
the large layer's H and I, `reps` times.  Device memory stays at a few GB so a
full Nsight Compute capture of one launch ends quickly; inputs still exceed L2.

    python -m token_dispatch_grouped_topk_gb300.profile_case [--E 32] [--rows 512]
           [--H 7168] [--I 2048] [--reps 3]
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
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    E, R, H, I = a.E, a.rows, a.H, a.I
    recv = W.activations(E * R, H, 1, dev).view(E, R, H)
    counts = torch.full((E,), R, dtype=torch.int32, device=dev)
    w13, s13, w2, s2 = W.expert_weights(E, H, I, 2, dev)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    out = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    times = {"quant": [], "gemm_gateup": [], "gemm_down": []}
    for _ in range(a.reps):
        ev[0].record()
        xq, xs = api.moe_quantize_fp8(recv, counts)
        ev[1].record()
        zq, zs = api.moe_gemm_gateup_silu(xq, xs, counts, w13, s13, dev_status=st)
        ev[2].record()
        api.moe_gemm_down(zq, zs, counts, w2, s2, out=out, dev_status=st)
        ev[3].record()
        torch.cuda.synchronize()
        for j, k in enumerate(times):
            times[k].append(ev[j].elapsed_time(ev[j + 1]))
    s = st.cpu().tolist()
    if s != [0, 0]:
        raise SystemExit(f"device status {s}")
    rows = E * R
    best = {k: min(v[1:] or v) for k, v in times.items()}
    print(f"profile case ok: E={E} rows={R} H={H} I={I} reps={a.reps}; best ms "
          + ", ".join(f"{k} {v:.4f}" for k, v in best.items())
          + f"; gate/up {4.0 * rows * H * I / best['gemm_gateup'] / 1e9:.1f} TFLOP/s"
          + f", down {2.0 * rows * H * I / best['gemm_down'] / 1e9:.1f} TFLOP/s")


if __name__ == "__main__":
    main()
