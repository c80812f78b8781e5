"""Shared test helpers: tensor conversion, the tolerance metric and oracle
calls on GPU-produced or GPU-consumed tensors."""
import numpy as np
import torch

import oracle as O

REL_TOL = 2e-2   # max relative error per row vs the fp64 oracle on the same quantised operands


def f32(t: torch.Tensor) -> np.ndarray:
    """Any float tensor (bf16 included) to a numpy fp32 array on the host."""
    return t.detach().to("cpu", torch.float32).numpy()


def u8(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    return t.detach().cpu().numpy()


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per row: max_h |got - ref| / max_h |ref|.  Rows whose reference is all
    zero must be exactly zero (returned as 0 or inf)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref), axis=1)
    num = np.max(np.abs(got - ref), axis=1)
    out = np.where(den > 0, num / np.where(den > 0, den, 1.0), np.where(num == 0, 0.0, np.inf))
    return out


def assert_rows_close(got, ref, tol=REL_TOL, what="rows"):
    err = row_rel_err(got, ref)
    assert np.all(np.isfinite(np.asarray(got))), f"{what}: non-finite values"
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max row relative error {worst:.3e} > {tol}"
    return worst


def host_weights(d, experts):
    """Host numpy copies of the given experts' weights and scales."""
    out = {}
    for e in experts:
        out[e] = (u8(d["w13"][e]), f32(d["s13"][e]), u8(d["w2"][e]), f32(d["s2"][e]))
    return out


def oracle_expert_rows(x_rows: np.ndarray, wts) -> np.ndarray:
    """fp64 oracle expert output for fp32 (bf16-valued) input rows."""
    xq, sx = O.quantize_rows(x_rows)
    w13, s13, w2, s2 = wts
    return O.expert_forward(xq, sx, w13, s13, w2, s2)[0]
