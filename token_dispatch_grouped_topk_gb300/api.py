"""Python entry points with the names of the C ABI (``include/moe.h``).

PyTorch supplies device memory, tensors' ``data_ptr()`` and the current CUDA
stream; every computation runs in the library's sm_103a kernels.  Outputs not
passed in are allocated with torch on the input's device.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib

__all__ = [
    "MoeError", "dispatch_workspace_size", "expert_compute_workspace_size",
    "expert_compute_workspace_layout", "moe_dispatch",
    "moe_dispatch_quant",
    "moe_expert_compute", "moe_combine", "moe_quantize_fp8", "moe_gemm_gateup_silu",
    "moe_gemm_down", "moe_gemm_gateup_down", "moe_dispatch_packed", "moe_expert_compute_packed",
    "moe_combine_packed", "moe_dispatch_source_slots", "moe_expert_compute_source_slots",
    "moe_dispatch_quant_source_slots", "moe_gemm_source_slots",
    "moe_layer_stats", "layer_stats_dict", "LAYER_STATS",
    "packed_rows", "MoeLayerBuffers", "HostPipeline", "TwoBatchOverlap", "DEV_BAD_EXPERT_ID",
    "DEV_CAPACITY_DROPPED", "DEV_TIMEOUT",
]

MoeError = _lib.MoeError
DEV_BAD_EXPERT_ID = _lib.DEV_BAD_EXPERT_ID
DEV_CAPACITY_DROPPED = _lib.DEV_CAPACITY_DROPPED
DEV_TIMEOUT = _lib.DEV_TIMEOUT


def _p(t):
    return None if t is None else t.data_ptr()


def _s(stream):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _u8(t):
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def dispatch_workspace_size(T: int, K: int, E: int) -> int:
    return int(_lib.load().moe_dispatch_workspace_size(T, K, E))


def expert_compute_workspace_size(E: int, R: int, H: int, I: int) -> int:
    return int(_lib.load().moe_expert_compute_workspace_size(E, R, H, I))


def expert_compute_workspace_layout(E: int, R: int, rows: int, H: int, I: int) -> list:
    """Byte offsets [xq, xs, zq, zs, sync, sync bytes, total] of the expert
    compute workspace, as the library carves it (rows = 0: padded layout)."""
    off = (ctypes.c_size_t * 7)()
    _lib.check("moe_expert_compute_workspace_layout",
               _lib.load().moe_expert_compute_workspace_layout(E, R, rows, H, I, off))
    return [int(v) for v in off]


def _workspace(nbytes, device):
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _gemm_flags(w13_interleaved, gemm_launch, max_ctas=0):
    """Flags of the GEMM launch form: None = the library's choice by tile
    count, "one" = both GEMMs in one launch, "two" = gate/up then down;
    max_ctas > 0 caps the GEMMs' persistent grid (MOE_GEMM_MAX_CTAS)."""
    f = _lib.W13_INTERLEAVED if w13_interleaved else 0
    if not 0 <= max_ctas <= 0x7FFF:
        raise ValueError("max_ctas must be in [0, 32767]")
    f |= max_ctas << 16
    if gemm_launch == "one":
        return f | _lib.GEMM_ONE_LAUNCH
    if gemm_launch == "two":
        return f | _lib.GEMM_TWO_LAUNCHES
    if gemm_launch is not None:
        raise ValueError(f"gemm_launch: None, 'one' or 'two', not {gemm_launch!r}")
    return f


def _idx_bits(topk_idx):
    """Router ids may be int64 or int32 (moe_dispatch_ex)."""
    if topk_idx.dtype == torch.int64:
        return 64
    if topk_idx.dtype == torch.int32:
        return 32
    raise TypeError(f"topk_idx: expected int64 or int32, got {topk_idx.dtype}")


def moe_dispatch(x, topk_idx, topk_w, E: int, R: int, *, recv=None, counts=None, src_map=None,
                 dev_status=None, workspace=None, stream=None):
    """Top-k dispatch into the expert-major receive buffer; ``topk_idx`` int64
    or int32.  Returns ``(recv [E,R,H] bf16, counts [E] int32, src_map [T,K]
    int32, dev_status [2] int32)``."""
    lib = _lib.load()
    T, H = x.shape
    K = topk_idx.shape[1]
    dev = x.device
    _need(x, torch.bfloat16, "x")
    bits = _idx_bits(topk_idx)
    _need(topk_idx, topk_idx.dtype, "topk_idx")
    if recv is None:
        recv = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if src_map is None:
        src_map = torch.empty(T, K, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_dispatch_workspace_size(T, K, E), dev)
    st = lib.moe_dispatch_ex(_p(x), _p(topk_idx), bits, _p(topk_w), T, H, K, E, R, 0, _p(recv),
                             _p(counts), _p(src_map), _p(dev_status), _p(workspace),
                             workspace.numel(), _s(stream))
    _lib.check("moe_dispatch_ex", st)
    return recv, counts, src_map, dev_status


def moe_dispatch_quant(x, topk_idx, topk_w, E: int, R: int, *, xq=None, xs=None, counts=None,
                       src_map=None, dev_status=None, workspace=None, stream=None, rows=0):
    """Dispatch fused with the per-token FP8 quantisation (moe_dispatch_quant_ex);
    ``topk_idx`` int64 or int32.  ``rows = 0``: padded layout, ``xq [E,R,H]``;
    ``rows > 0``: packed layout, ``xq [rows,H]``.  Returns ``(xq uint8, xs
    fp32, counts, src_map, dev_status)``."""
    lib = _lib.load()
    T, H = x.shape
    K = topk_idx.shape[1]
    dev = x.device
    _need(x, torch.bfloat16, "x")
    bits = _idx_bits(topk_idx)
    _need(topk_idx, topk_idx.dtype, "topk_idx")
    lead = (rows,) if rows else (E, R)
    if xq is None:
        xq = torch.empty(*lead, H, dtype=torch.uint8, device=dev)
    if xs is None:
        xs = torch.empty(*lead, H // 128, dtype=torch.float32, device=dev)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if src_map is None:
        src_map = torch.empty(T, K, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_dispatch_workspace_size(T, K, E), dev)
    st = lib.moe_dispatch_quant_ex(_p(x), _p(topk_idx), bits, _p(topk_w), T, H, K, E, R, rows,
                                   _p(_u8(xq)), _p(xs), _p(counts), _p(src_map), _p(dev_status),
                                   _p(workspace), workspace.numel(), _s(stream))
    _lib.check("moe_dispatch_quant_ex", st)
    return xq, xs, counts, src_map, dev_status


def moe_expert_compute(recv, counts, w13, w13_scale, w2, w2_scale, *, out=None, dev_status=None,
                       workspace=None, stream=None, w13_interleaved=False, gemm_launch=None,
                       max_ctas=0):
    """Quantise the valid rows and run the grouped gated-SiLU FP8 expert MLP.
    Returns ``out [E,R,H] bf16`` (rows past counts[e] untouched).  With
    ``w13_interleaved`` the W13 rows alternate gate and up (moe_expert_compute_ex)."""
    lib = _lib.load()
    E, R, H = recv.shape
    w13, w2 = _u8(w13), _u8(w2)
    I = w13.shape[1] // 2
    dev = recv.device
    if out is None:
        out = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_expert_compute_workspace_size(E, R, H, I), dev)
    st = lib.moe_expert_compute_ex(_p(recv), _p(counts), E, R, 0, H, I, _p(w13), _p(w13_scale),
                                   _p(w2), _p(w2_scale), _p(out), _p(dev_status), _p(workspace),
                                   workspace.numel(),
                                   _gemm_flags(w13_interleaved, gemm_launch, max_ctas), _s(stream))
    _lib.check("moe_expert_compute_ex", st)
    return out


def moe_dispatch_source_slots(x, topk_idx, topk_w, E: int, L: int, max_tokens: int, *,
                              rank_offsets=None, recv=None, counts=None, seg_counts=None,
                              src_map=None, dev_status=None, stream=None):
    """Dispatch into the per-source fixed-slot layout (moe_dispatch_source_slots):
    expert e's W*max_tokens rows hold one range of max_tokens slots per source
    rank.  Returns ``(recv [E, W*max_tokens, H] bf16, counts [E], seg_counts
    [E, W], src_map [T, K], dev_status)``."""
    lib = _lib.load()
    T, H = x.shape
    K = topk_idx.shape[1]
    W = E // L
    dev = x.device
    _need(x, torch.bfloat16, "x")
    bits = _idx_bits(topk_idx)
    _need(topk_idx, topk_idx.dtype, "topk_idx")
    if recv is None:
        recv = torch.empty(E, W * max_tokens, H, dtype=torch.bfloat16, device=dev)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if seg_counts is None:
        seg_counts = torch.empty(E, W, dtype=torch.int32, device=dev)
    if src_map is None:
        src_map = torch.empty(T, K, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(2, dtype=torch.int32, device=dev)
    st = lib.moe_dispatch_source_slots(_p(x), _p(topk_idx), bits, _p(topk_w), T, H, K, E, L,
                                       max_tokens, _p(rank_offsets), _p(recv), _p(counts),
                                       _p(seg_counts), _p(src_map), _p(dev_status), _s(stream))
    _lib.check("moe_dispatch_source_slots", st)
    return recv, counts, seg_counts, src_map, dev_status


def moe_expert_compute_source_slots(recv, counts, seg_counts, L: int, max_tokens: int, w13,
                                    w13_scale, w2, w2_scale, *, out=None, dev_status=None,
                                    workspace=None, stream=None, w13_interleaved=False,
                                    gemm_launch=None):
    """``moe_expert_compute`` on the per-source fixed-slot layout: only the rows
    that hold a route are quantised and stored.  Returns ``out [E, W*max_tokens,
    H] bf16`` (other rows untouched)."""
    lib = _lib.load()
    E, R, H = recv.shape
    w13, w2 = _u8(w13), _u8(w2)
    I = w13.shape[1] // 2
    dev = recv.device
    if out is None:
        out = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_expert_compute_workspace_size(E, R, H, I), dev)
    st = lib.moe_expert_compute_source_slots(
        _p(recv), _p(counts), _p(seg_counts), E, L, max_tokens, H, I, _p(w13), _p(w13_scale),
        _p(w2), _p(w2_scale), _p(out), _p(dev_status), _p(workspace), workspace.numel(),
        _gemm_flags(w13_interleaved, gemm_launch), _s(stream))
    _lib.check("moe_expert_compute_source_slots", st)
    return out


def moe_dispatch_quant_source_slots(x, topk_idx, topk_w, E: int, L: int, max_tokens: int, *,
                                    rank_offsets=None, xq=None, xs=None, counts=None,
                                    seg_counts=None, src_map=None, dev_status=None, stream=None):
    """``moe_dispatch_source_slots`` fused with the per-token FP8 quantisation:
    each token row is quantised once and its codes and scales are written to
    every kept slot.  Returns ``(xq [E, W*max_tokens, H] uint8, xs [E,
    W*max_tokens, H/128] fp32, counts, seg_counts, src_map, dev_status)``."""
    lib = _lib.load()
    T, H = x.shape
    K = topk_idx.shape[1]
    W = E // L
    dev = x.device
    _need(x, torch.bfloat16, "x")
    bits = _idx_bits(topk_idx)
    _need(topk_idx, topk_idx.dtype, "topk_idx")
    if xq is None:
        xq = torch.empty(E, W * max_tokens, H, dtype=torch.uint8, device=dev)
    if xs is None:
        xs = torch.empty(E, W * max_tokens, H // 128, dtype=torch.float32, device=dev)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if seg_counts is None:
        seg_counts = torch.empty(E, W, dtype=torch.int32, device=dev)
    if src_map is None:
        src_map = torch.empty(T, K, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(2, dtype=torch.int32, device=dev)
    st = lib.moe_dispatch_quant_source_slots(
        _p(x), _p(topk_idx), bits, _p(topk_w), T, H, K, E, L, max_tokens, _p(rank_offsets),
        _p(_u8(xq)), _p(xs), _p(counts), _p(seg_counts), _p(src_map), _p(dev_status), _s(stream))
    _lib.check("moe_dispatch_quant_source_slots", st)
    return xq, xs, counts, seg_counts, src_map, dev_status


def moe_gemm_source_slots(xq, xs, seg_counts, L: int, max_tokens: int, w13, w13_scale, w2,
                          w2_scale, *, out=None, dev_status=None, workspace=None, stream=None,
                          w13_interleaved=False, gemm_launch=None, max_ctas=0):
    """Both GEMMs on the FP8 slots of ``moe_dispatch_quant_source_slots``: the
    valid rows are packed in the workspace, then the GEMMs of
    ``moe_expert_compute_source_slots`` run.  Returns ``out [E, W*max_tokens, H]
    bf16`` (other rows untouched)."""
    lib = _lib.load()
    xq = _u8(xq)
    E, R, H = xq.shape
    w13, w2 = _u8(w13), _u8(w2)
    I = w13.shape[1] // 2
    dev = xq.device
    if out is None:
        out = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_expert_compute_workspace_size(E, R, H, I), dev)
    st = lib.moe_gemm_source_slots(
        _p(xq), _p(xs), _p(seg_counts), E, L, max_tokens, H, I, _p(w13), _p(w13_scale), _p(w2),
        _p(w2_scale), _p(out), _p(dev_status), _p(workspace), workspace.numel(),
        _gemm_flags(w13_interleaved, gemm_launch, max_ctas), _s(stream))
    _lib.check("moe_gemm_source_slots", st)
    return out


def packed_rows(T: int, K: int, E: int, R: int) -> int:
    """Rows of a packed receive buffer with room for every kept route:
    min(T*K, E*R) ("SGLang Expert Compute Backend", §2.6)."""
    return max(1, min(T * K, E * R))


def moe_dispatch_packed(x, topk_idx, topk_w, E: int, R: int, *, rows=None, recv=None, counts=None,
                        src_map=None, dev_status=None, workspace=None, stream=None):
    """Dispatch into the packed layout: expert e's rows back to back from the
    prefix of the clamped counts.  Returns ``(recv [rows,H] bf16, counts,
    src_map (= base_e + slot), dev_status)``."""
    lib = _lib.load()
    T, H = x.shape
    K = topk_idx.shape[1]
    dev = x.device
    _need(x, torch.bfloat16, "x")
    bits = _idx_bits(topk_idx)
    _need(topk_idx, topk_idx.dtype, "topk_idx")
    if rows is None:
        rows = recv.shape[0] if recv is not None else packed_rows(T, K, E, R)
    if recv is None:
        recv = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if src_map is None:
        src_map = torch.empty(T, K, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_dispatch_workspace_size(T, K, E), dev)
    st = lib.moe_dispatch_ex(_p(x), _p(topk_idx), bits, _p(topk_w), T, H, K, E, R, rows, _p(recv),
                             _p(counts), _p(src_map), _p(dev_status), _p(workspace),
                             workspace.numel(), _s(stream))
    _lib.check("moe_dispatch_ex", st)
    return recv, counts, src_map, dev_status


def moe_expert_compute_packed(recv, counts, R: int, w13, w13_scale, w2, w2_scale, *, out=None,
                              dev_status=None, workspace=None, stream=None, w13_interleaved=False,
                              gemm_launch=None):
    """``moe_expert_compute`` on the packed layout: recv and out are [rows, H]."""
    lib = _lib.load()
    rows, H = recv.shape
    E = counts.shape[0]
    w13, w2 = _u8(w13), _u8(w2)
    I = w13.shape[1] // 2
    dev = recv.device
    if out is None:
        out = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(lib.moe_expert_compute_packed_workspace_size(rows, H, I), dev)
    st = lib.moe_expert_compute_ex(_p(recv), _p(counts), E, R, rows, H, I, _p(w13), _p(w13_scale),
                                   _p(w2), _p(w2_scale), _p(out), _p(dev_status), _p(workspace),
                                   workspace.numel(), _gemm_flags(w13_interleaved, gemm_launch),
                                   _s(stream))
    _lib.check("moe_expert_compute_ex", st)
    return out


LAYER_STATS = ("valid_routes", "kept_routes", "messages", "cross_rank_routes", "tile_blocks",
               "active_experts", "busiest_expert_rows")


def moe_layer_stats(topk_idx, counts, L: int, R: int, *, rank_offsets=None, stats=None,
                    stream=None):
    """Route, message and tile counts of one routing (moe_layer_stats); returns
    the device ``stats`` tensor (int64 [7], in the order of ``LAYER_STATS``)."""
    lib = _lib.load()
    T, K = topk_idx.shape
    E = counts.shape[0]
    if stats is None:
        stats = torch.empty(len(LAYER_STATS), dtype=torch.int64, device=counts.device)
    st = lib.moe_layer_stats(_p(topk_idx), _idx_bits(topk_idx), _p(counts), T, K, E, L, R,
                             _p(rank_offsets), _p(stats), _s(stream))
    _lib.check("moe_layer_stats", st)
    return stats


def layer_stats_dict(stats, E: int, R: int) -> dict:
    """Host view of moe_layer_stats' counters, with the derived figures:
    dropped routes, M-row fill of the 128-row blocks, and the blocks a
    capacity-dense launch would cover."""
    v = [int(x) for x in stats.cpu().tolist()]
    d = dict(zip(LAYER_STATS, v))
    d["dropped_routes"] = d["valid_routes"] - d["kept_routes"]
    d["m_fill_128"] = d["kept_routes"] / (128 * d["tile_blocks"]) if d["tile_blocks"] else None
    d["capacity_blocks"] = E * -(-R // 128)
    return d


def moe_combine_packed(out, src_map, topk_w, *, y=None, stream=None):
    """``moe_combine`` on the packed layout: out is [rows, H]."""
    lib = _lib.load()
    rows, H = out.shape
    T, K = src_map.shape
    if y is None:
        y = torch.empty(T, H, dtype=torch.bfloat16, device=out.device)
    st = lib.moe_combine_packed(_p(out), rows, _p(src_map), _p(topk_w), T, H, K, _p(y), _s(stream))
    _lib.check("moe_combine_packed", st)
    return y


def moe_combine(out, src_map, topk_w, *, y=None, stream=None):
    """Weighted combine back into token order.  Returns ``y [T,H] bf16``."""
    lib = _lib.load()
    E, R, H = out.shape
    T, K = src_map.shape
    if y is None:
        y = torch.empty(T, H, dtype=torch.bfloat16, device=out.device)
    st = lib.moe_combine(_p(out), _p(src_map), _p(topk_w), T, H, K, E, R, _p(y), _s(stream))
    _lib.check("moe_combine", st)
    return y


def moe_quantize_fp8(recv, counts, *, xq=None, xs=None, stream=None):
    """Per-token FP8 quantisation of the valid rows: ``xq [E,R,H] uint8`` (e4m3
    codes) and ``xs [E,R,H/128] fp32``."""
    lib = _lib.load()
    E, R, H = recv.shape
    if xq is None:
        xq = torch.empty(E, R, H, dtype=torch.uint8, device=recv.device)
    if xs is None:
        xs = torch.empty(E, R, H // 128, dtype=torch.float32, device=recv.device)
    st = lib.moe_quantize_fp8(_p(recv), _p(counts), E, R, H, _p(xq), _p(xs), _s(stream))
    _lib.check("moe_quantize_fp8", st)
    return xq, xs


def moe_gemm_gateup_silu(xq, xs, counts, w13, w13_scale, *, zq=None, zs=None, dev_status=None,
                         stream=None):
    """Gate/up GEMM + SiLU(gate)*up + FP8 requant: ``zq [E,R,I]``, ``zs [E,R,I/128]``."""
    lib = _lib.load()
    E, R, H = xq.shape
    w13 = _u8(w13)
    I = w13.shape[1] // 2
    dev = xq.device
    if zq is None:
        zq = torch.empty(E, R, I, dtype=torch.uint8, device=dev)
    if zs is None:
        zs = torch.empty(E, R, I // 128, dtype=torch.float32, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    st = lib.moe_gemm_gateup_silu(_p(_u8(xq)), _p(xs), _p(counts), E, R, H, I, _p(w13),
                                  _p(w13_scale), _p(zq), _p(zs), _p(dev_status), _s(stream))
    _lib.check("moe_gemm_gateup_silu", st)
    return zq, zs


def moe_gemm_down(zq, zs, counts, w2, w2_scale, *, out=None, dev_status=None, stream=None):
    """Down GEMM: ``out [E,R,H] bf16`` for the valid rows."""
    lib = _lib.load()
    E, R, I = zq.shape
    w2 = _u8(w2)
    H = w2.shape[1]
    dev = zq.device
    if out is None:
        out = torch.empty(E, R, H, dtype=torch.bfloat16, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    st = lib.moe_gemm_down(_p(_u8(zq)), _p(zs), _p(counts), E, R, H, I, _p(w2), _p(w2_scale),
                           _p(out), _p(dev_status), _s(stream))
    _lib.check("moe_gemm_down", st)
    return out


def moe_gemm_gateup_down(xq, xs, counts, w13, w13_scale, w2, w2_scale, *, R=None, zq=None,
                         zs=None, out=None, sync=None, dev_status=None, stream=None,
                         w13_interleaved=False, gemm_launch=None, max_ctas=0):
    """Both GEMMs in one launch (down tiles start per 128-row block as soon as
    that block's Z is written); bit-identical to ``moe_gemm_gateup_silu`` then
    ``moe_gemm_down``.  ``xq [E,R,H]`` is the padded layout; ``xq [rows,H]``
    with ``R`` given is the packed one.  Returns ``out``."""
    lib = _lib.load()
    w13, w2 = _u8(w13), _u8(w2)
    E = counts.shape[0]
    I = w13.shape[1] // 2
    dev = xq.device
    if xq.dim() == 3:
        E, R, H = xq.shape
        rows, lead = 0, (E, R)
    else:
        if R is None:
            raise ValueError("the packed layout needs R")
        rows, H = xq.shape
        lead = (rows,)
    if zq is None:
        zq = torch.empty(*lead, I, dtype=torch.uint8, device=dev)
    if zs is None:
        zs = torch.empty(*lead, I // 128, dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty(*lead, H, dtype=torch.bfloat16, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
    if sync is None:
        sync = _workspace(lib.moe_gemm_gateup_down_sync_size(E, R, rows), dev)
    st = lib.moe_gemm_gateup_down(_p(_u8(xq)), _p(xs), _p(counts), E, R, rows, H, I, _p(w13),
                                  _p(w13_scale), _p(w2), _p(w2_scale), _p(zq), _p(zs), _p(out),
                                  _p(dev_status), _p(sync), sync.numel() * sync.element_size(),
                                  _gemm_flags(w13_interleaved, gemm_launch, max_ctas), _s(stream))
    _lib.check("moe_gemm_gateup_down", st)
    return out


@dataclass
class MoeLayerBuffers:
    """One resource set ("lane") for a routed MoE layer: every buffer the three
    calls touch, allocated once so the calls can be repeated or captured into a
    CUDA graph.  Two instances give the two independent lanes a two-micro-batch
    split needs ("SGLang、NCCL 与 MoE EP", §2.4: each micro-batch owns its own
    receive, routing and output storage)."""

    T: int
    E: int
    K: int
    H: int
    I: int
    R: int
    device: torch.device
    packed: bool = False   # packed layout (moe_*_packed): [rows, H] buffers, no capacity gaps
    w13_interleaved: bool = False   # W13 rows alternate gate and up
    gemm_launch: str | None = None  # None: the library's choice; "one" / "two" launches
    # per-source fixed slots (moe_*_source_slots): max tokens per source rank
    # (0: off); then R must be (E / L) * source_slots, rank_offsets optional
    source_slots: int = 0
    L: int = 1
    rank_offsets: torch.Tensor | None = None

    def __post_init__(self):
        d, E, R, H, I, T, K = self.device, self.E, self.R, self.H, self.I, self.T, self.K
        if self.source_slots:
            if self.packed or E % self.L or R != (E // self.L) * self.source_slots:
                raise ValueError("source slots: padded lane with R = (E / L) * max_tokens")
            self.seg_counts = torch.zeros(E, E // self.L, dtype=torch.int32, device=d)
        if self.packed:
            self.rows = packed_rows(T, K, E, R)
            shape = (self.rows, H)
            ws = _lib.load().moe_expert_compute_packed_workspace_size(self.rows, H, I)
        else:
            self.rows = E * R
            shape = (E, R, H)
            ws = expert_compute_workspace_size(E, R, H, I)
        self._recv_shape = shape
        self._recv = None
        self._slots = None
        self.out = torch.empty(*shape, dtype=torch.bfloat16, device=d)
        self.counts = torch.zeros(E, dtype=torch.int32, device=d)
        self.src_map = torch.empty(T, K, dtype=torch.int32, device=d)
        self.dev_status = torch.zeros(2, dtype=torch.int32, device=d)
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=d)
        self.ws_dispatch = _workspace(dispatch_workspace_size(T, K, E), d)
        self.ws_compute = _workspace(ws, d)

    @property
    def recv(self):
        """The BF16 receive buffer of the separate path, allocated on first
        use (the default fused path never forms it: 15 GB saved at the large
        padded layer).  Touch it before capturing a separate-path forward into
        a CUDA graph."""
        if self._recv is None:
            self._recv = torch.empty(*self._recv_shape, dtype=torch.bfloat16, device=self.device)
        return self._recv

    @property
    def slots_fp8(self):
        """(xq [E, R, H] uint8, xs [E, R, H/128] fp32): the FP8 slots the fused
        path of the per-source layout dispatches into (the expert compute packs
        their valid rows into its workspace), allocated on first use.  Touch it
        before capturing a fused forward of a per-source lane into a CUDA
        graph."""
        if self._slots is None:
            E, R, H = self.E, self.R, self.H
            self._slots = (torch.empty(E, R, H, dtype=torch.uint8, device=self.device),
                           torch.empty(E, R, H // 128, dtype=torch.float32, device=self.device))
        return self._slots

    def workspace_layout(self):
        """Byte offsets of the expert compute workspace's parts, from the
        library (moe_expert_compute_workspace_layout): xq, xs, zq, zs, sync,
        sync bytes, total."""
        return expert_compute_workspace_layout(self.E, self.R, self.rows if self.packed else 0,
                                               self.H, self.I)

    def workspace_views(self):
        """(xq, xs, zq, zs): the FP8 activations and scales inside the expert
        compute workspace, in the layout moe_expert_compute(_packed) uses:
        [E, R, ...] padded, [rows, ...] packed."""
        H, I, n = self.H, self.I, self.rows
        lead = (self.rows,) if self.packed else (self.E, self.R)
        G, GI = H // 128, I // 128
        o = self.workspace_layout()
        ws = self.ws_compute
        xq = ws[o[0]:o[0] + n * H].view(*lead, H)
        xs = ws[o[1]:o[1] + n * G * 4].view(torch.float32).view(*lead, G)
        zq = ws[o[2]:o[2] + n * I].view(*lead, I)
        zs = ws[o[3]:o[3] + n * GI * 4].view(torch.float32).view(*lead, GI)
        return xq, xs, zq, zs

    def sync_view(self):
        """The fused GEMM launch's scratch inside the expert compute workspace
        (a tile ticket and one count per 128-row block)."""
        o = self.workspace_layout()
        return self.ws_compute[o[4]:o[4] + o[5]]

    def dispatch_quant(self, x, topk_idx, topk_w, stream=None):
        """The layer's first stage on the fused path: moe_dispatch_quant_ex
        into the workspace's FP8 activations (the BF16 receive buffer is not
        used); on the per-source layout moe_dispatch_quant_source_slots into
        ``slots_fp8``."""
        if self.source_slots:
            sq, ss = self.slots_fp8
            moe_dispatch_quant_source_slots(x, topk_idx, topk_w, self.E, self.L,
                                            self.source_slots, rank_offsets=self.rank_offsets,
                                            xq=sq, xs=ss, counts=self.counts,
                                            seg_counts=self.seg_counts, src_map=self.src_map,
                                            dev_status=self.dev_status, stream=stream)
            return
        xq, xs, _, _ = self.workspace_views()
        moe_dispatch_quant(x, topk_idx, topk_w, self.E, self.R, xq=xq, xs=xs, counts=self.counts,
                           src_map=self.src_map, dev_status=self.dev_status,
                           workspace=self.ws_dispatch, stream=stream,
                           rows=self.rows if self.packed else 0)

    def gemms(self, w13, w13_scale, w2, w2_scale, stream=None, max_ctas=0):
        """Both GEMMs on the FP8 activations dispatch_quant wrote, in the
        library's launch form for the layer (or ``gemm_launch``)."""
        if self.source_slots:
            sq, ss = self.slots_fp8
            moe_gemm_source_slots(sq, ss, self.seg_counts, self.L, self.source_slots, w13,
                                  w13_scale, w2, w2_scale, out=self.out,
                                  dev_status=self.dev_status, workspace=self.ws_compute,
                                  stream=stream, w13_interleaved=self.w13_interleaved,
                                  gemm_launch=self.gemm_launch, max_ctas=max_ctas)
            return
        xq, xs, zq, zs = self.workspace_views()
        moe_gemm_gateup_down(xq, xs, self.counts, w13, w13_scale, w2, w2_scale, R=self.R, zq=zq,
                             zs=zs, out=self.out, sync=self.sync_view(), dev_status=self.dev_status,
                             stream=stream, w13_interleaved=self.w13_interleaved,
                             gemm_launch=self.gemm_launch, max_ctas=max_ctas)

    def combine(self, topk_w, y, stream=None):
        if self.packed:
            moe_combine_packed(self.out, self.src_map, topk_w, y=y, stream=stream)
        else:
            moe_combine(self.out, self.src_map, topk_w, y=y, stream=stream)

    def forward_fused(self, x, topk_idx, topk_w, w13, w13_scale, w2, w2_scale, stream=None, y=None):
        """``forward(..., fused=True)``."""
        return self.forward(x, topk_idx, topk_w, w13, w13_scale, w2, w2_scale, stream=stream, y=y,
                            fused=True)

    def forward(self, x, topk_idx, topk_w, w13, w13_scale, w2, w2_scale, stream=None, y=None,
                fused=None):
        """The layer on one stream; returns ``y`` (the lane's own output buffer
        unless ``y`` [T, H] BF16 is given).

        ``fused`` None or True: dispatch fused with the quantisation (each
        token row quantised once, FP8 rows scattered; on the per-source layout
        into ``slots_fp8``) -> both GEMMs -> combine; the faster path on the
        padded and packed layouts, by 4-7 % per layer step on GB300, and on
        the per-source layout 1 % faster at decode with 18 % less lane
        memory.  ``fused=False``: dispatch of BF16 rows into ``recv`` ->
        expert compute (quantisation, GEMMs) -> combine.  Both give the same
        ``y``, bit for bit."""
        y = self.y if y is None else y
        if fused is None or fused:
            self.dispatch_quant(x, topk_idx, topk_w, stream=stream)
            self.gemms(w13, w13_scale, w2, w2_scale, stream=stream)
            self.combine(topk_w, y, stream=stream)
            return y
        if self.source_slots:
            moe_dispatch_source_slots(x, topk_idx, topk_w, self.E, self.L, self.source_slots,
                                      rank_offsets=self.rank_offsets, recv=self.recv,
                                      counts=self.counts, seg_counts=self.seg_counts,
                                      src_map=self.src_map, dev_status=self.dev_status,
                                      stream=stream)
            moe_expert_compute_source_slots(self.recv, self.counts, self.seg_counts, self.L,
                                            self.source_slots, w13, w13_scale, w2, w2_scale,
                                            out=self.out, dev_status=self.dev_status,
                                            workspace=self.ws_compute, stream=stream,
                                            w13_interleaved=self.w13_interleaved,
                                            gemm_launch=self.gemm_launch)
            moe_combine(self.out, self.src_map, topk_w, y=y, stream=stream)
            return y
        if self.packed:
            moe_dispatch_packed(x, topk_idx, topk_w, self.E, self.R, recv=self.recv,
                                counts=self.counts, src_map=self.src_map,
                                dev_status=self.dev_status, workspace=self.ws_dispatch,
                                stream=stream)
            moe_expert_compute_packed(self.recv, self.counts, self.R, w13, w13_scale, w2,
                                      w2_scale, out=self.out, dev_status=self.dev_status,
                                      workspace=self.ws_compute, stream=stream,
                                      w13_interleaved=self.w13_interleaved,
                                      gemm_launch=self.gemm_launch)
            moe_combine_packed(self.out, self.src_map, topk_w, y=y, stream=stream)
            return y
        moe_dispatch(x, topk_idx, topk_w, self.E, self.R, recv=self.recv, counts=self.counts,
                     src_map=self.src_map, dev_status=self.dev_status, workspace=self.ws_dispatch,
                     stream=stream)
        moe_expert_compute(self.recv, self.counts, w13, w13_scale, w2, w2_scale, out=self.out,
                           dev_status=self.dev_status, workspace=self.ws_compute, stream=stream,
                           w13_interleaved=self.w13_interleaved, gemm_launch=self.gemm_launch)
        moe_combine(self.out, self.src_map, topk_w, y=y, stream=stream)
        return y


class HostPipeline:
    """Layer invocations fed from pinned host memory and returned to it, with
    the copies of neighbouring steps overlapped with compute: while step i
    computes on the caller's stream, step i+1's inputs are copied in on one
    copy stream and step i-1's output is copied out on another.  Inputs and
    outputs have two device slots each; events order every reuse of a slot
    (a slot is refilled only after the compute that read it, and an output
    slot is rewritten only after its copy to the host).  The layer itself runs
    on one buffer lane, in submission order.  Host tensors must be pinned and
    must not be touched until ``synchronize()`` (or a later step's completion)
    has returned.

    With ``graph=True`` the layer of each input slot is captured once into a
    CUDA graph (on the slot's first step, which runs eagerly) and replayed on
    later steps, so a step costs one graph launch instead of the layer's
    separate launches.  A graph is kept per slot and set of weight tensors;
    new weight tensors are captured anew."""

    def __init__(self, lane: "MoeLayerBuffers", graph: bool = False):
        self.lane = lane
        self.graph = graph
        self._graphs = {}
        d, T, H, K = lane.device, lane.T, lane.H, lane.K
        self.x = [torch.empty(T, H, dtype=torch.bfloat16, device=d) for _ in range(2)]
        self.idx = [torch.empty(T, K, dtype=torch.int64, device=d) for _ in range(2)]
        self.w = [torch.empty(T, K, dtype=torch.float32, device=d) for _ in range(2)]
        self.y = [torch.empty(T, H, dtype=torch.bfloat16, device=d) for _ in range(2)]
        self.s_in = torch.cuda.Stream(d)
        self.s_out = torch.cuda.Stream(d)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.in_ready, self.in_free, self.y_ready, self.y_free = ev(), ev(), ev(), ev()
        self.n = 0

    def submit(self, x_h, idx_h, w_h, y_h, w13, w13_scale, w2, w2_scale, stream=None):
        """Queue one layer step: x_h [T, H] BF16, idx_h [T, K] int64 and w_h
        [T, K] fp32 (pinned host) in, y_h [T, H] BF16 (pinned host) out."""
        for t in (x_h, idx_h, w_h, y_h):
            if t.is_cuda or not t.is_pinned():
                raise ValueError("HostPipeline takes pinned host tensors")
        k = self.n % 2
        cs = stream if stream is not None else torch.cuda.current_stream(self.lane.device)
        if self.n >= 2:
            self.s_in.wait_event(self.in_free[k])
        with torch.cuda.stream(self.s_in):
            self.x[k].copy_(x_h, non_blocking=True)
            self.idx[k].copy_(idx_h, non_blocking=True)
            self.w[k].copy_(w_h, non_blocking=True)
        self.in_ready[k].record(self.s_in)
        cs.wait_event(self.in_ready[k])
        if self.n >= 2:
            cs.wait_event(self.y_free[k])
        self._compute(k, (w13, w13_scale, w2, w2_scale), cs)
        self.in_free[k].record(cs)
        self.y_ready[k].record(cs)
        self.s_out.wait_event(self.y_ready[k])
        with torch.cuda.stream(self.s_out):
            y_h.copy_(self.y[k], non_blocking=True)
        self.y_free[k].record(self.s_out)
        self.n += 1

    def _forward(self, k, weights, stream):
        self.lane.forward(self.x[k], self.idx[k], self.w[k], *weights, stream=stream, y=self.y[k])

    def _compute(self, k, weights, cs):
        if not self.graph:
            self._forward(k, weights, cs)
            return
        key = (k,) + tuple(t.data_ptr() for t in weights)
        g = self._graphs.get(key)
        if g is None:
            # this step runs eagerly; the capture records the same launches
            # without running them
            self._forward(k, weights, cs)
            side = torch.cuda.Stream(self.lane.device)
            side.wait_stream(cs)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self._forward(k, weights, side)
            cs.wait_stream(side)
            self._graphs[key] = g
            return
        with torch.cuda.stream(cs):
            g.replay()

    def synchronize(self):
        """Wait until every submitted step's output is in host memory."""
        self.s_out.synchronize()


class TwoBatchOverlap:
    """A layer split into two micro-batches (token halves), each with its own
    buffer lane, on two CUDA streams: micro-batch B's dispatch runs beside A's
    expert compute and B's expert compute beside A's combine ("SGLang、NCCL 与
    MoE EP", §2.4 and §5.4: two-batch overlap needs one resource set per
    micro-batch; the overlap can at best hide min(D, S) of the two stages).
    ``forward(..., overlap=False)`` runs the same two halves back to back on
    one stream (the "serial split" of "SGLang Expert Compute Backend", §5.6).
    Both produce the same bytes.  The stages are those of
    ``MoeLayerBuffers.forward``: with ``fused`` (default) dispatch+quantisation,
    GEMMs, combine; without, dispatch, expert compute (quantisation and GEMMs),
    combine."""

    def __init__(self, T: int, E: int, K: int, H: int, I: int, R: int, device, gemm_ctas: int = 0,
                 fused: bool = True):
        self.gemm_ctas = gemm_ctas   # > 0: the expert compute's GEMMs take at most this many SMs
        self.fused = fused
        self.half = T // 2
        self.sizes = (self.half, T - self.half)
        self.lanes = [MoeLayerBuffers(n, E, K, H, I, R, device) for n in self.sizes]
        self.streams = [torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)]
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        # each lane's combine writes straight into its half of y
        self.lanes[0].y = self.y[: self.half]
        self.lanes[1].y = self.y[self.half:]
        self.ev = [torch.cuda.Event() for _ in range(2)]

    def _views(self, x, topk_idx, topk_w):
        h = self.half
        return [(x[:h], topk_idx[:h], topk_w[:h]), (x[h:], topk_idx[h:], topk_w[h:])]

    def _stage(self, lane, name, inp, weights, stream):
        x, idx, w = inp
        if self.fused:
            if name == "dispatch":
                lane.dispatch_quant(x, idx, w, stream=stream)
            elif name == "compute":
                lane.gemms(*weights, stream=stream, max_ctas=self.gemm_ctas)
            else:
                lane.combine(w, lane.y, stream=stream)
            return
        if name == "dispatch":
            moe_dispatch(x, idx, w, lane.E, lane.R, recv=lane.recv, counts=lane.counts,
                         src_map=lane.src_map, dev_status=lane.dev_status,
                         workspace=lane.ws_dispatch, stream=stream)
        elif name == "compute":
            moe_expert_compute(lane.recv, lane.counts, *weights, out=lane.out,
                               dev_status=lane.dev_status, workspace=lane.ws_compute, stream=stream,
                               max_ctas=self.gemm_ctas)
        else:
            moe_combine(lane.out, lane.src_map, w, y=lane.y, stream=stream)

    def forward(self, x, topk_idx, topk_w, w13, w13_scale, w2, w2_scale, overlap: bool = True):
        weights = (w13, w13_scale, w2, w2_scale)
        views = self._views(x, topk_idx, topk_w)
        cur = torch.cuda.current_stream()
        a, b = self.lanes
        if not overlap:
            for lane, v in zip(self.lanes, views):
                for name in ("dispatch", "compute", "combine"):
                    self._stage(lane, name, v, weights, cur)
        else:
            sa, sb = self.streams
            sa.wait_stream(cur)
            sb.wait_stream(cur)
            self._stage(a, "dispatch", views[0], weights, sa)
            self.ev[0].record(sa)
            self._stage(a, "compute", views[0], weights, sa)
            self.ev[1].record(sa)
            sb.wait_event(self.ev[0])            # B's dispatch beside A's expert compute
            self._stage(b, "dispatch", views[1], weights, sb)
            self._stage(a, "combine", views[0], weights, sa)
            sb.wait_event(self.ev[1])            # B's expert compute beside A's combine
            self._stage(b, "compute", views[1], weights, sb)
            self._stage(b, "combine", views[1], weights, sb)
            cur.wait_stream(sa)
            cur.wait_stream(sb)
        return self.y
