"""Seeded synthetic inputs for the routed MoE branch.

This module only draws random inputs; it holds none of the layer's arithmetic.
Both the CUDA path and the CPU oracle are fed from here.

Workloads (shapes from the pages' traced scenario and GEMM example, plus three
larger synthetic layers):

* ``traced``   -- "SGLang、NCCL 与 MoE EP", problem two: 4 logical EP ranks, 8
  experts (2 per rank), top-2, local tokens [0, 16, 32, 64]; rank 2 token 5
  picks E1, E6 at weights 0.25 / 0.75, every other token E0, E7 at w, 1-w.
* ``gemm_unit`` -- "SGLang Expert Compute Backend", §2.3: 2 local experts,
  receive buffer [2, 128, 256] with valid counts [70, 12], H=256, I=128.
* ``decode``   -- T=256, E=64 (8x8), top-8, H=4096, I=1536, R=256.
* ``prefill``  -- T=4096, E=128 (16x8), top-8, H=4096, I=1536, R=2048, Zipf(1.1)
  expert popularity added to the router logits; also run as two micro-batches
  of 2048 tokens.
* ``large``    -- T=16384, E=256 (32x8), top-8, H=7168, I=2048, R=4096, per-expert
  logit bias ~ N(0, 0.5).

Activations are BF16 ~ N(0, 1).  Master weights are fp32 ~ N(0, 0.02), stored as
e4m3 codes with one fp32 scale per 128x128 block (scale = block amax / 448, the
codes produced by PyTorch's own e4m3 cast), so dequantised values follow
N(0, 0.02).  Router: logits ~ N(0, 1) plus the workload's bias, top-K of the
biased logits, weights = softmax over the K selected logits.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # total tokens, logical ranks concatenated in rank order
    E: int            # global experts
    W: int            # logical EP ranks (E = W * L)
    K: int            # top-k
    H: int            # hidden size
    I: int            # expert intermediate size
    R: int            # capacity rows per expert
    bias: str = "none"           # router logit bias: none | zipf | normal
    tokens_per_rank: tuple = field(default=())

    @property
    def L(self) -> int:
        return self.E // self.W


WORKLOADS = {
    "traced": Workload("traced", T=112, E=8, W=4, K=2, H=256, I=128, R=128,
                       tokens_per_rank=(0, 16, 32, 64)),
    "gemm_unit": Workload("gemm_unit", T=0, E=2, W=1, K=1, H=256, I=128, R=128),
    "decode": Workload("decode", T=256, E=64, W=8, K=8, H=4096, I=1536, R=256),
    "prefill": Workload("prefill", T=4096, E=128, W=16, K=8, H=4096, I=1536, R=2048, bias="zipf"),
    "large": Workload("large", T=16384, E=256, W=32, K=8, H=7168, I=2048, R=4096, bias="normal"),
}

GEMM_UNIT_COUNTS = (70, 12)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def activations(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """BF16 activations ~ N(0, 1), [T, H]."""
    g = _gen(seed, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def block_fp8_weights(E: int, N: int, Kd: int, seed: int, device="cpu", std: float = 0.02):
    """Expert weights stored [E, N, Kd] as e4m3 codes (uint8) plus fp32 scales
    [E, N/128, Kd/128], one per 128x128 block.  Generated expert by expert to
    bound peak memory."""
    g = _gen(seed, device)
    codes = torch.empty(E, N, Kd, dtype=torch.uint8, device=device)
    scales = torch.empty(E, N // 128, Kd // 128, dtype=torch.float32, device=device)
    for e in range(E):
        w = torch.randn(N, Kd, generator=g, device=device, dtype=torch.float32) * std
        blk = w.view(N // 128, 128, Kd // 128, 128)
        amax = blk.abs().amax(dim=(1, 3))
        s = amax / 448.0
        q = (blk / s[:, None, :, None]).to(torch.float8_e4m3fn)
        codes[e] = q.view(N, Kd).view(torch.uint8)
        scales[e] = s
    return codes, scales


def expert_weights(E: int, H: int, I: int, seed: int, device="cpu"):
    """(w13 [E, 2I, H], s13 [E, 2I/128, H/128], w2 [E, H, I], s2 [E, H/128, I/128])."""
    w13, s13 = block_fp8_weights(E, 2 * I, H, seed * 2 + 1, device)
    w2, s2 = block_fp8_weights(E, H, I, seed * 2 + 2, device)
    return w13, s13, w2, s2


def router_bias(wl: Workload, seed: int, device="cpu") -> torch.Tensor:
    E = wl.E
    g = _gen(seed + 7919, "cpu")
    if wl.bias == "zipf":
        ranks = torch.randperm(E, generator=g).to(torch.float64) + 1.0
        p = ranks ** -1.1
        p = p / p.sum()
        return torch.log(p).to(torch.float32).to(device)
    if wl.bias == "normal":
        return (torch.randn(E, generator=g, dtype=torch.float32) * 0.5).to(device)
    return torch.zeros(E, dtype=torch.float32, device=device)


def router(T: int, E: int, K: int, bias: torch.Tensor, seed: int, device="cpu"):
    """Top-K of biased N(0,1) logits; weights = softmax over the K selected
    logits.  Returns (topk_idx int64 [T, K], topk_w fp32 [T, K])."""
    g = _gen(seed, device)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32) + bias.to(device)
    vals, idx = torch.topk(logits, K, dim=1)
    w = torch.softmax(vals, dim=1)
    return idx.to(torch.int64).contiguous(), w.to(torch.float32).contiguous()


def traced_routes(seed: int = 0, swap_token_21: bool = False):
    """The pages' hand-traced routing.  Global token 21 (rank 2, row 5) picks
    E1, E6 at 0.25 / 0.75 (or E0, E7 for the replay of §3.4); every other
    token picks E0, E7 at w, 1-w with w ~ U(0, 1)."""
    wl = WORKLOADS["traced"]
    g = _gen(seed, "cpu")
    w = torch.rand(wl.T, generator=g, dtype=torch.float32)
    idx = torch.tensor([[0, 7]] * wl.T, dtype=torch.int64)
    topk_w = torch.stack([w, 1.0 - w], dim=1)
    t21 = sum(wl.tokens_per_rank[:2]) + 5
    idx[t21] = torch.tensor([0, 7] if swap_token_21 else [1, 6])
    topk_w[t21] = torch.tensor([0.25, 0.75])
    return idx, topk_w.contiguous()


def source_rank_of_tokens(wl: Workload) -> torch.Tensor:
    """Logical source rank of each global token (ranks concatenated in order).
    Workloads without an explicit split use T/W tokens per rank."""
    per = wl.tokens_per_rank or tuple([wl.T // wl.W] * wl.W)
    return torch.repeat_interleave(torch.arange(len(per)), torch.tensor(per))


def make_layer_inputs(name: str, seed: int = 0, device="cpu", weights: bool = True):
    """All inputs of one layer invocation of a named workload (not gemm_unit)."""
    wl = WORKLOADS[name]
    if name == "traced":
        idx, w = traced_routes(seed)
        idx, w = idx.to(device), w.to(device)
    else:
        idx, w = router(wl.T, wl.E, wl.K, router_bias(wl, seed, device), seed + 1, device)
    out = {"wl": wl, "x": activations(wl.T, wl.H, seed + 2, device), "topk_idx": idx, "topk_w": w}
    if weights:
        out["w13"], out["s13"], out["w2"], out["s2"] = expert_weights(wl.E, wl.H, wl.I, seed + 3, device)
    return out


def gemm_unit_inputs(seed: int = 0, device="cpu"):
    """Receive buffer [2, 128, 256] BF16 with valid prefixes [70, 12]; the
    capacity rows past each count are filled with NaN so any read of them shows
    up in the outputs."""
    wl = WORKLOADS["gemm_unit"]
    recv = torch.full((wl.E, wl.R, wl.H), float("nan"), dtype=torch.bfloat16, device=device)
    x = activations(sum(GEMM_UNIT_COUNTS), wl.H, seed, device)
    off = 0
    for e, c in enumerate(GEMM_UNIT_COUNTS):
        recv[e, :c] = x[off:off + c]
        off += c
    counts = torch.tensor(GEMM_UNIT_COUNTS, dtype=torch.int32, device=device)
    w13, s13, w2, s2 = expert_weights(wl.E, wl.H, wl.I, seed + 3, device)
    return {"wl": wl, "recv": recv, "counts": counts, "w13": w13, "s13": s13, "w2": w2, "s2": s2}
