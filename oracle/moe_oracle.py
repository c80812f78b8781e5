"""Plain, slow, obviously-correct CPU oracle for one MoE layer's routed branch.

TEST INFRASTRUCTURE ONLY -- imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  It
shares no code with the CUDA path.  Floating point is fp64 except where the
method itself fixes fp32 (the quantisation rule and the combine restatement).

Each function names the passage it follows as "<page title>, <section>".
Readings taken where the pages are silent or garbled:

* within-expert slot order: the pages leave it to atomic arrival order
  ("SGLang、NCCL 与 MoE EP", §2.3.4: any order is a valid compact prefix).  The
  oracle fixes the canonical order -- ascending route id ``i = t*K + k`` -- so
  layouts compare bit for bit; the tests also check the order-free property.
* capacity overflow: the pages assume capacity always covers the routes.  When
  it does not, routes past ``R`` (in canonical order) are dropped: their source
  map entry is -1, they are counted in ``dropped`` and excluded from combine.
* the combine restatement used for bit-exact GPU checks accumulates in fp32 in
  ascending k, one multiply and one add per term (two roundings), starting at 0,
  then rounds to BF16 to nearest even.
* SiLU(g) = g / (1 + exp(-g)); gate/up are not interleaved (first I columns are
  gate, the last I are up).

Parity pins (``tests/test_oracle_pins.py``) tie every function here to values
the pages print or to closed forms / library routines; see that file.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

QUANT_GROUP = 128          # one scale per row per 128 hidden elements
E4M3_MAX = 448.0           # largest finite e4m3 magnitude
AMAX_FLOOR = np.float32(1e-4)

__all__ = [
    "QUANT_GROUP", "E4M3_MAX",
    "e4m3_decode", "e4m3_encode", "bf16_bits_to_f32", "f32_to_bf16_rne",
    "f32_to_bf16_bits", "expert_placement", "RouteResult", "route", "scatter",
    "packed_row_offsets", "packed_src_map", "SourceSlotResult", "route_source_slots",
    "route_stats", "quantize_rows", "gemm_block_scaled", "silu",
    "expert_forward", "combine_fp64", "combine_f32_sequential", "moe_layer",
    "m_blocks", "valid_tiles", "m_fill_rate", "align_index_capacity",
    "align_grid", "row_major_offset",
]


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def _e4m3_table() -> np.ndarray:
    """Value of each of the 256 e4m3 (``float8_e4m3fn``) codes.

    OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits; exponent field 0 is subnormal with step 2**-9; there is no
    infinity and S.1111.111 is NaN; the largest finite magnitude is 448.
    """
    table = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man = code & 0x7
        if exp_field == 0xF and man == 0x7:
            table[code] = math.nan
        elif exp_field == 0:
            table[code] = sign * man * 2.0 ** -9
        else:
            table[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return table


_E4M3 = _e4m3_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Decode e4m3 codes (uint8) to fp64 values."""
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Encode finite fp32 values to e4m3 codes, round-to-nearest-even, saturating
    to +-448 ("satfinite").

    The value is rounded to a multiple of the quantum of its binade: 2**(e-3)
    for |v| in [2**e, 2**(e+1)) with e >= -6, and the subnormal step 2**-9
    below 2**-6.  ``np.rint`` rounds halves to even, which for a quotient by a
    power of two is round-to-nearest-even on the mantissa.
    """
    v = np.asarray(v, dtype=np.float32)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3_encode: non-finite input")
    a = np.abs(v).astype(np.float64)
    neg = np.signbit(v)
    _, ex = np.frexp(a)                      # a = m * 2**ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)               # binade exponent; subnormals share 2**-6's quantum
    quantum = np.ldexp(1.0, e - 3)
    val = np.rint(a / quantum) * quantum     # exact in fp64
    val = np.minimum(val, E4M3_MAX)          # satfinite
    code = np.zeros(a.shape, dtype=np.int64)
    sub = val < 2.0 ** -6
    code[sub] = (val[sub] / 2.0 ** -9).astype(np.int64)          # exponent field 0
    nrm = ~sub
    _, ex2 = np.frexp(val[nrm])
    e2 = ex2 - 1
    man = (val[nrm] / np.ldexp(1.0, e2) - 1.0) * 8.0
    code[nrm] = ((e2 + 7) << 3) | man.astype(np.int64)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) to the fp32 values they denote (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 to BF16 (nearest, ties to even) and return the bit patterns.

    BF16 keeps the top 16 bits of the fp32 pattern; adding 0x7FFF plus the
    lowest kept bit before truncation rounds to nearest with ties to even.
    Inputs must be finite.
    """
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def f32_to_bf16_rne(v: np.ndarray) -> np.ndarray:
    """fp32 -> nearest BF16 value (ties to even), returned as fp32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(v))


# ---------------------------------------------------------------------------
# Routing: placement, count + slot assignment, scatter
# ---------------------------------------------------------------------------

def expert_placement(g: int, L: int) -> tuple[int, int]:
    """Global expert g lives on logical rank g // L as local expert g % L
    ("SGLang、NCCL 与 MoE EP", §2.1, contiguous even split L = E / W)."""
    return g // L, g % L


@dataclass
class RouteResult:
    counts: np.ndarray        # [E] int32, kept rows per expert (<= R)
    src_map: np.ndarray       # [T, K] int32, flat row q = e*R + s, or -1
    routed: np.ndarray        # [E] int64, routes per expert before capacity
    dropped: int              # routes past capacity
    bad_id: bool              # some id outside [-1, E)


def route(topk_idx: np.ndarray, E: int, R: int) -> RouteResult:
    """Count and slot assignment of every route.

    "SGLang、NCCL 与 MoE EP", §2.3.4: each route to expert e takes the next row
    s of that expert's counter (the counter is also the row allocator), writes
    its payload to ``recv[e, s]`` and records the flat row ``q = e*M + s``
    (§2.3.6).  Ids of -1 are padding routes (§2.3.1).  Slots are handed out in
    ascending route id i = t*K + k (canonical order, see module docstring);
    routes past capacity R are dropped.
    """
    topk_idx = np.asarray(topk_idx)
    T, K = topk_idx.shape
    fill = np.zeros(E, dtype=np.int64)
    src_map = np.full((T, K), -1, dtype=np.int32)
    dropped = 0
    bad = False
    ids = topk_idx.tolist()
    for t in range(T):
        row = ids[t]
        for k in range(K):
            e = int(row[k])
            if e == -1:
                continue
            if e < -1 or e >= E:
                bad = True
                continue
            s = int(fill[e])
            fill[e] += 1
            if s < R:
                src_map[t, k] = e * R + s
            else:
                dropped += 1
    counts = np.minimum(fill, R).astype(np.int32)
    return RouteResult(counts=counts, src_map=src_map, routed=fill, dropped=dropped, bad_id=bad)


def scatter(x: np.ndarray, src_map: np.ndarray, E: int, R: int) -> np.ndarray:
    """``recv[e, s, :] = x[t, :]`` for every kept route ("SGLang、NCCL 与 MoE EP",
    §2.3.4).  Rows that receive nothing are NaN (they are capacity padding and
    must not be read)."""
    T, H = x.shape
    recv = np.full((E * R, H), np.nan, dtype=x.dtype)
    for t in range(T):
        for q in src_map[t]:
            if q >= 0:
                recv[q] = x[t]
    return recv.reshape(E, R, H)


def packed_row_offsets(counts) -> np.ndarray:
    """Compact storage, "SGLang Expert Compute Backend", §2.6: the valid rows
    of the experts are laid out back to back, so expert e starts where expert
    e-1's valid rows end.  Returns the E+1 offsets (offsets[-1] = total valid
    rows).  In the page's example, counts [70, 12] put expert 1's first row
    right after expert 0's 70th: offsets [0, 70, 82]."""
    off = [0]
    for c in counts:
        off.append(off[-1] + int(c))
    return np.asarray(off, dtype=np.int64)


def packed_src_map(src_map: np.ndarray, counts, R: int) -> np.ndarray:
    """The source map of the packed layout: route (t, k) kept at slot s of
    expert e (flat padded row q = e*R + s) is stored at row offsets[e] + s."""
    off = packed_row_offsets(counts)
    out = np.full_like(src_map, -1)
    for idx, q in np.ndenumerate(src_map):
        if q >= 0:
            e, s = divmod(int(q), R)
            out[idx] = off[e] + s
    return out


@dataclass
class SourceSlotResult:
    counts: np.ndarray        # [E] int32, valid rows per expert (masked_m)
    seg_counts: np.ndarray    # [E, W] int32, valid rows per (expert, source rank)
    src_map: np.ndarray       # [T, K] int32, q = e*W*max_tokens + r*max_tokens + p, or -1
    dropped: int              # routes past their source's slot range
    bad_id: bool              # some id outside [-1, E)


def route_source_slots(topk_idx: np.ndarray, E: int, L: int, max_tokens: int,
                       src_rank: np.ndarray) -> SourceSlotResult:
    """The low-latency receive layout of "DeepEP 架构与实现笔记", §9.5: the
    receive buffer is [L, W*max_tokens, H] and every source rank owns a fixed
    range of max_tokens slots inside every expert, so a route's row follows
    from its source rank r and its position p among r's routes to that expert
    -- row r*max_tokens + p -- with no layout agreed across ranks first.  Valid
    rows are therefore not one prefix per expert: each (expert, source) range
    holds its own valid count, and the rows between are padding.  Positions
    are taken in ascending route id (the canonical order of ``route``); a route
    whose position reaches max_tokens has no slot and is dropped.  Here the
    experts of all ranks share one buffer [E, W*max_tokens, H], so the flat
    row is q = e*W*max_tokens + r*max_tokens + p."""
    topk_idx = np.asarray(topk_idx)
    T, K = topk_idx.shape
    W = E // L
    R = W * max_tokens
    fill = np.zeros((E, W), dtype=np.int64)
    src_map = np.full((T, K), -1, dtype=np.int32)
    dropped = 0
    bad = False
    ids = topk_idx.tolist()
    for t in range(T):
        r = int(src_rank[t])
        for k in range(K):
            e = int(ids[t][k])
            if e == -1:
                continue
            if e < -1 or e >= E:
                bad = True
                continue
            p = int(fill[e, r])
            fill[e, r] += 1
            if p < max_tokens:
                src_map[t, k] = e * R + r * max_tokens + p
            else:
                dropped += 1
    seg = np.minimum(fill, max_tokens).astype(np.int32)
    return SourceSlotResult(counts=seg.sum(axis=1).astype(np.int32), seg_counts=seg,
                            src_map=src_map, dropped=dropped, bad_id=bad)


def route_stats(topk_idx: np.ndarray, L: int, src_rank: np.ndarray) -> dict:
    """Byte-accounting counts of "SGLang、NCCL 与 MoE EP", §5.3.

    ``messages`` = sum over tokens of D_t, the number of distinct destination
    ranks among the token's valid routes (one payload per destination rank,
    §2.3.2); ``cross_rank_routes`` = routes whose destination rank differs
    from the token's source rank; ``routes`` = sum of valid routes.
    """
    topk_idx = np.asarray(topk_idx)
    messages = 0
    routes = 0
    cross = 0
    for t in range(topk_idx.shape[0]):
        dests = set()
        for e in topk_idx[t]:
            e = int(e)
            if e < 0:
                continue
            r, _ = expert_placement(e, L)
            dests.add(r)
            routes += 1
            if r != int(src_rank[t]):
                cross += 1
        messages += len(dests)
    return {"messages": messages, "routes": routes, "cross_rank_routes": cross}


# ---------------------------------------------------------------------------
# Per-token FP8 quantisation
# ---------------------------------------------------------------------------

def quantize_rows(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-row, per-128-element FP8 quantisation.

    "DeepEP 架构与实现笔记", §11: per token and per 128 hidden elements take
    amax = max|v| clamped below at 1e-4, scale the block by 448/amax into the
    e4m3 range, cast to e4m3, and keep the fp32 scale amax/448.  The receive
    side applies it to every valid row ("SGLang、NCCL 与 MoE EP", §2.3.5: FP32
    scales of shape [L, M, H/128]).  All arithmetic is fp32 as the rule states
    (fp32 division and multiply, each rounded to nearest).
    """
    v = np.asarray(v, dtype=np.float32)
    rows, H = v.shape
    if H % QUANT_GROUP:
        raise ValueError("hidden size must be a multiple of 128")
    blocks = v.reshape(rows, H // QUANT_GROUP, QUANT_GROUP)
    amax = np.max(np.abs(blocks), axis=2) if rows else np.zeros((0, H // QUANT_GROUP), np.float32)
    amax = np.maximum(amax, AMAX_FLOOR).astype(np.float32)
    ratio = (np.float32(E4M3_MAX) / amax).astype(np.float32)
    scaled = (blocks * ratio[:, :, None]).astype(np.float32)
    codes = e4m3_encode(scaled).reshape(rows, H)
    scales = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return codes, scales


# ---------------------------------------------------------------------------
# Gated-SiLU expert
# ---------------------------------------------------------------------------

def gemm_block_scaled(aq: np.ndarray, sa: np.ndarray, wq: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """Block-scaled FP8 GEMM, fp64.

    "SGLang Expert Compute Backend", §3.5: activations carry one scale per row
    per 128 K-elements, weights (stored [N, K], output-major) one scale per
    128x128 (N, K) block; the product is the sum over K-groups g of
    ``sa[m, g] * sw[n // 128, g] * sum_{k in g} a[m, k] * w[n, k]``.
    """
    m, K = aq.shape
    N = wq.shape[0]
    A = e4m3_decode(aq)
    W = e4m3_decode(wq)
    out = np.zeros((m, N), dtype=np.float64)
    for g in range(K // QUANT_GROUP):
        ks = slice(g * QUANT_GROUP, (g + 1) * QUANT_GROUP)
        part = A[:, ks] @ W[:, ks].T
        col_scale = np.repeat(sw[:, g].astype(np.float64), QUANT_GROUP)[:N]
        out += sa[:, g].astype(np.float64)[:, None] * col_scale[None, :] * part
    return out


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g)), fp64."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def expert_forward(xq, sx, w13q, s13, w2q, s2, interleaved: bool = False):
    """One expert on its valid rows.

    "SGLang Expert Compute Backend", §1.1: X[m,H] -> gate/up GEMM [m, 2I] ->
    SiLU(gate) * up [m, I] -> down GEMM [m, H]; §3.6: the first I columns are
    gate and the last I are up, and the down input is re-quantised per row per
    128 like the activations.  With ``interleaved`` the gate/up weight rows
    alternate instead ("XTuner Domino EP", complete runtime path: SiLU of the
    even output columns times the odd ones).  G and Z are fp64; Z is taken to
    fp32 before the fp32 quantisation rule.  Returns ``(out, zq, sz, G)``.
    """
    I = w13q.shape[0] // 2
    G = gemm_block_scaled(xq, sx, w13q, s13)
    if interleaved:
        Z = silu(G[:, 0::2]) * G[:, 1::2]
    else:
        Z = silu(G[:, :I]) * G[:, I:]
    zq, sz = quantize_rows(Z.astype(np.float32))
    out = gemm_block_scaled(zq, sz, w2q, s2)
    return out, zq, sz, G


# ---------------------------------------------------------------------------
# Combine
# ---------------------------------------------------------------------------

def combine_fp64(route_out: np.ndarray, src_map: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """``y[t] = sum_k w[t, k] * out[q(t, k)]`` over kept routes, fp64.

    "SGLang、NCCL 与 MoE EP", §1.1 (the routed output sum, weights on the
    expert output) and §3.2 (each route's output multiplied by its weight
    exactly once and summed into the token's own row).  ``route_out`` is
    indexed by flat row q.
    """
    T, K = src_map.shape
    H = route_out.shape[1]
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for k in range(K):
            q = int(src_map[t, k])
            if q >= 0:
                y[t] += float(topk_w[t, k]) * route_out[q].astype(np.float64)
    return y


def combine_f32_sequential(out_flat: np.ndarray, src_map: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """Combine restated in fp32 for bit-exact comparison: ``acc = 0``; for k
    ascending over kept routes ``acc = acc + w[t,k] * out[q]`` with the product
    and the sum each rounded to fp32; the result rounded to BF16 (nearest
    even).  Returned as fp32 values."""
    T, K = src_map.shape
    H = out_flat.shape[1]
    acc = np.zeros((T, H), dtype=np.float32)
    w = np.asarray(topk_w, dtype=np.float32)
    for k in range(K):
        q = src_map[:, k]
        m = q >= 0
        prod = (w[m, k][:, None] * out_flat[q[m]].astype(np.float32)).astype(np.float32)
        acc[m] = (acc[m] + prod).astype(np.float32)
    return f32_to_bf16_rne(acc)


# ---------------------------------------------------------------------------
# Whole layer (independent reference enumerating the original ids)
# ---------------------------------------------------------------------------

def moe_layer(x, topk_idx, topk_w, w13q, s13, w2q, s2, E: int, R: int):
    """The routed branch end to end, fp64.

    Following "SGLang、NCCL 与 MoE EP", §5.1, the reference walks each source
    token's experts from the original ids instead of reusing the dispatcher's
    map: ``y[t] = sum_k w[t,k] * F_e(quant(x[t]))`` over the routes kept by
    capacity.  Per-row quantisation does not depend on the slot, so each token
    is quantised once.  Returns ``(y, RouteResult, route_out)`` where
    ``route_out[t, k]`` is the expert output of route (t, k) (zeros if the
    route is not kept).
    """
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    K = topk_idx.shape[1]
    rr = route(topk_idx, E, R)
    xq, sx = quantize_rows(x)
    route_out = np.zeros((T, K, H), dtype=np.float64)
    for e in range(E):
        tk = np.argwhere((np.asarray(topk_idx) == e) & (rr.src_map >= 0))
        if len(tk) == 0:
            continue
        toks = tk[:, 0]
        out, _, _, _ = expert_forward(xq[toks], sx[toks], w13q[e], s13[e], w2q[e], s2[e])
        route_out[tk[:, 0], tk[:, 1]] = out
    w = np.where(rr.src_map >= 0, np.asarray(topk_w, dtype=np.float64), 0.0)
    y = np.einsum("tk,tkh->th", w, route_out)
    return y, rr, route_out


# ---------------------------------------------------------------------------
# Tile counting and the addressing of the worked [70, 12] example
# ---------------------------------------------------------------------------

def m_blocks(counts, BM: int) -> int:
    """Valid M-blocks when every expert is tiled on its own:
    sum_e ceil(m_e / BM) ("SGLang Expert Compute Backend", §2.4, §4.3)."""
    return int(sum(-(-int(c) // BM) for c in counts))


def valid_tiles(counts, BM: int, BN: int, N: int) -> int:
    """Valid output tiles: sum_e ceil(m_e/BM) * ceil(N/BN) (§2.4 of the same
    page: 6 tiles for counts [70, 12] at BM64, BN128, N=256)."""
    return m_blocks(counts, BM) * -(-N // BN)


def m_fill_rate(counts, BM: int) -> float:
    """M-row fill rate sum m_e / (BM * sum ceil(m_e/BM)) ("SGLang Expert
    Compute Backend", §5.4); only defined for a non-zero denominator."""
    blocks = m_blocks(counts, BM)
    return float(sum(int(c) for c in counts)) / (BM * blocks)


def align_index_capacity(S: int, L: int, BM: int) -> int:
    """Index capacity Q of the alignment step the reference backend runs before
    its grouped GEMM ("SGLang Expert Compute Backend", §3.3): S + (L+1)(BM-1)
    when S >= L+1, else S*BM.  Kept only to cross-check tile counting."""
    return S + (L + 1) * (BM - 1) if S >= L + 1 else S * BM


def align_grid(S: int, L: int, BM: int, BN: int, N: int) -> int:
    """Programs that backend launches per GEMM: ceil(Q/BM) * ceil(N/BN)
    (§3.4 and the §4.3 table of the same page)."""
    Q = align_index_capacity(S, L, BM)
    return -(-Q // BM) * -(-N // BN)


def row_major_offset(shape, index) -> int:
    """Element offset of ``index`` in a contiguous row-major tensor."""
    off = 0
    for dim, i in zip(shape, index):
        if not 0 <= i < dim:
            raise IndexError(index)
        off = off * dim + i
    return off
