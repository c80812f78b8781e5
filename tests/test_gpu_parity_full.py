"""Whole-config parity of the layer at the prefill and large shapes.

The prefill-shaped layer (T=4096, E=128, H=4096, I=1536, R=2048) is checked on
every kept route; the large layer (T=16384, E=256, H=7168, I=2048, R=4096) on
every kept route of at least 16 whole experts chosen to cover the busiest
expert, the lightest active ones and every size class of an expert's last
128-row block (1-32, 33-64, 65-127 and 128 rows).  Each expert output row is
compared with the fp64 oracle on the same quantised operands (max relative
error per row <= 2e-2), the combine with the fp32 restatement (bit-exact, every
token), and the layer output y with the fp64 oracle where all of a token's
routes were computed by it.

For the worst row of each config the error is split in two by recomputing the
down GEMM in the oracle from the GPU's own Z codes and scales: what the down
GEMM adds (fp32 accumulation and the BF16 rounding of the output) and what
comes from Z itself (Z codes one e4m3 step away from the oracle's where the
fp32 gate/up accumulation lands on the other side of a rounding midpoint).

Setting MOE_PARITY_REPORT=<path> writes the per-config figures as JSON.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_grouped_topk_gb300 import api
from token_dispatch_grouped_topk_gb300 import workloads as W

from helpers import REL_TOL, f32, host_weights, row_rel_err, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
_REPORT = {}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api._lib.load()
    yield
    torch.cuda.synchronize()
    path = os.environ.get("MOE_PARITY_REPORT")
    if path and _REPORT:
        with open(path, "w") as f:
            json.dump(_REPORT, f, indent=1)


def _run_layer(name, seed):
    d = W.make_layer_inputs(name, seed=seed, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    buf.forward(d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    torch.cuda.synchronize()
    assert buf.dev_status[0].item() & api.DEV_TIMEOUT == 0
    rr = O.route(d["topk_idx"].cpu().numpy(), wl.E, wl.R)
    assert buf.counts.cpu().numpy().tolist() == rr.counts.tolist()
    assert np.array_equal(buf.src_map.cpu().numpy(), rr.src_map)
    return d, wl, buf, rr


def _e4m3_step_distance(a_codes, b_codes):
    """Number of e4m3 steps between two code arrays of the same sign class
    (codes of one sign are ordered by magnitude)."""
    a = a_codes.astype(np.int64)
    b = b_codes.astype(np.int64)
    sa, sb = a >> 7, b >> 7
    ma, mb = a & 0x7F, b & 0x7F
    same = sa == sb
    return np.where(same, np.abs(ma - mb), ma + mb)


def _check_experts(d, wl, buf, rr, experts):
    """Every kept route of `experts` against the oracle.  Returns the per-row
    errors, the oracle rows by flat row q, and the worst row's breakdown."""
    x = f32(d["x"])
    idx = d["topk_idx"].cpu().numpy()
    src = rr.src_map
    H, I = wl.H, wl.I
    out_flat = buf.out.view(-1, H)
    _, _, zq_ws, zs_ws = buf.workspace_views()
    zq_flat = zq_ws.reshape(-1, I)
    zs_flat = zs_ws.reshape(-1, I // 128)
    wts = host_weights(d, experts)
    errs, ref_rows = [], {}
    worst = (-1.0, None)
    for e in experts:
        tk = np.argwhere((idx == e) & (src >= 0))
        if len(tk) == 0:
            continue
        q = src[tk[:, 0], tk[:, 1]]
        order = np.argsort(q)                       # slot order
        tk, q = tk[order], q[order]
        w13, s13, w2, s2 = wts[e]
        xq, sx = O.quantize_rows(x[tk[:, 0]])
        ref, zq_ref, sz_ref, _ = O.expert_forward(xq, sx, w13, s13, w2, s2)
        got = f32(out_flat[torch.from_numpy(q).to(DEV).long()])
        err = row_rel_err(got, ref)
        assert np.all(np.isfinite(got)), f"expert {e}: non-finite rows"
        errs.append(err)
        for j, qq in enumerate(q):
            ref_rows[int(qq)] = ref[j]
        j = int(np.argmax(err))
        if err[j] > worst[0]:
            qj = int(q[j])
            zq_gpu = u8(zq_flat[qj])
            zs_gpu = f32(zs_flat[qj])
            via_gpu_z = O.gemm_block_scaled(zq_gpu[None, :], zs_gpu[None, :], w2, s2)[0]
            steps = _e4m3_step_distance(zq_gpu, zq_ref[j])
            worst = (float(err[j]), {
                "expert": int(e), "slot": int(qj - e * wl.R), "count": int(rr.counts[e]),
                "row_rel_err": float(err[j]),
                "down_gemm_part": float(row_rel_err(got[j:j + 1], via_gpu_z[None, :])[0]),
                "z_part": float(row_rel_err(via_gpu_z[None, :], ref[j:j + 1])[0]),
                "z_codes_differing": int(np.count_nonzero(steps)),
                "z_max_code_steps": int(steps.max()),
                "z_scale_max_rel_diff": float(np.max(np.abs(zs_gpu - sz_ref[j]) / sz_ref[j])),
            })
    return np.concatenate(errs), ref_rows, worst[1]


def _summary(errs, worst, extra):
    s = {"rows": int(errs.size), "worst": float(errs.max()), "p99_9": float(np.quantile(errs, 0.999)),
         "p99": float(np.quantile(errs, 0.99)), "median": float(np.median(errs)), "worst_row": worst}
    s.update(extra)
    return s


def _combine_all_tokens(wl, buf, rr, topk_w, chunk):
    """y of every token against the fp32 restatement, in token chunks."""
    y = f32(buf.y)
    H = wl.H
    w = topk_w.cpu().numpy()
    for t0 in range(0, wl.T, chunk):
        sm = rr.src_map[t0:t0 + chunk]
        uniq, inv = np.unique(sm[sm >= 0], return_inverse=True)
        compact = np.full_like(sm, -1)
        compact[sm >= 0] = inv
        rows = f32(buf.out.view(-1, H)[torch.from_numpy(uniq).to(DEV).long()])
        want = O.combine_f32_sequential(rows, compact, w[t0:t0 + chunk])
        assert np.array_equal(y[t0:t0 + chunk], want), f"combine differs in tokens [{t0}, {t0 + chunk})"
    return y


def test_prefill_every_kept_route():
    """Prefill-shaped Zipf-skewed layer: every kept route's expert output and
    every token's y against the fp64 oracle, combine bit-exact on every token."""
    d, wl, buf, rr = _run_layer("prefill", seed=0)
    experts = [e for e in range(wl.E) if rr.counts[e] > 0]
    errs, ref_rows, worst = _check_experts(d, wl, buf, rr, experts)
    assert errs.size == int(rr.counts.sum())
    y = _combine_all_tokens(wl, buf, rr, d["topk_w"], 1024)
    # y against the fp64 oracle: y_ref[t] = sum_k w[t,k] * out_ref[q(t,k)]
    w = d["topk_w"].cpu().numpy().astype(np.float64)
    y_ref = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        for k in range(wl.K):
            q = int(rr.src_map[t, k])
            if q >= 0:
                y_ref[t] += w[t, k] * ref_rows[q]
    yerr = row_rel_err(y, y_ref)
    _REPORT["prefill"] = _summary(errs, worst, {"experts": len(experts), "y_worst": float(yerr.max()),
                                                "y_p99_9": float(np.quantile(yerr, 0.999))})
    assert float(errs.max()) <= REL_TOL, _REPORT["prefill"]
    assert float(yerr.max()) <= REL_TOL, _REPORT["prefill"]


def _pick_large_experts(counts, rng):
    """At least 16 experts: the busiest, the three lightest active, two of
    each last-block size class, the rest at random."""
    c = np.asarray(counts)
    active = np.flatnonzero(c > 0)
    pick = [int(active[np.argmax(c[active])])]
    pick += [int(e) for e in active[np.argsort(c[active])[:3]]]
    tail = c % 128
    for lo, hi in ((1, 32), (33, 64), (65, 127), (0, 0)):
        cls = [int(e) for e in active if lo <= tail[e] <= hi and e not in pick]
        pick += [int(e) for e in rng.choice(cls, size=min(2, len(cls)), replace=False)] if cls else []
    rest = [int(e) for e in active if e not in pick]
    pick += [int(e) for e in rng.choice(rest, size=max(0, 16 - len(pick)), replace=False)]
    return sorted(set(pick))


def test_large_whole_experts():
    """Large layer: every kept route of >= 16 whole experts (busiest,
    lightest, each last-block size class) against the fp64 oracle; combine
    bit-exact on every token."""
    d, wl, buf, rr = _run_layer("large", seed=0)
    experts = _pick_large_experts(rr.counts, np.random.default_rng(5))
    assert len(experts) >= 16
    tails = {int(rr.counts[e]) % 128 for e in experts}
    assert any(1 <= t <= 32 for t in tails) and any(33 <= t <= 64 for t in tails)
    assert any(65 <= t <= 127 for t in tails)
    errs, _, worst = _check_experts(d, wl, buf, rr, experts)
    _combine_all_tokens(wl, buf, rr, d["topk_w"], 2048)
    _REPORT["large"] = _summary(errs, worst, {"experts": experts,
                                              "expert_counts": [int(rr.counts[e]) for e in experts]})
    assert float(errs.max()) <= REL_TOL, _REPORT["large"]


def test_worst_rows_are_explained_by_z_codes():
    """The worst row of each config, split: the down GEMM on the GPU's own Z
    adds no more than the BF16 output rounding and fp32 accumulation allow,
    so the rest of the row's error comes from Z codes (each at most one e4m3
    step from the oracle's)."""
    if not _REPORT:
        pytest.skip("runs after the whole-config tests of this file")
    for name, rep in _REPORT.items():
        w = rep["worst_row"]
        assert w["down_gemm_part"] <= 4e-3, (name, w)
        assert w["z_max_code_steps"] <= 1, (name, w)
