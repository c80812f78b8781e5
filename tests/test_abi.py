"""CPU checks of the C ABI: the library builds, loads, exports every entry
point include/moe.h declares, and rejects bad arguments on the host before
touching the GPU."""
import ctypes
import os
import re

import pytest
import torch

from token_dispatch_grouped_topk_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_calls():
    names = declared_functions()
    for fn in ("moe_dispatch", "moe_expert_compute", "moe_combine", "moe_dispatch_workspace_size",
               "moe_expert_compute_workspace_size", "moe_quantize_fp8", "moe_gemm_gateup_silu",
               "moe_gemm_down", "moe_abi_version", "moe_status_string"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_exports_are_c_symbols():
    out = os.popen(f"nm -D --defined-only {_lib._build.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (moe_\w+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_version_and_status_strings(lib):
    assert lib.moe_abi_version() == 1
    for code, name in _lib.STATUS.items():
        assert lib.moe_status_string(code).decode() == name


def test_workspace_sizes(lib):
    assert lib.moe_dispatch_workspace_size(-1, 2, 8) == 0
    assert lib.moe_dispatch_workspace_size(0, 2, 8) == 256
    # one int32 per (expert, block of 8 warps x 32/K tokens)
    assert lib.moe_dispatch_workspace_size(16384, 8, 256) == 256 * (16384 // 32) * 4
    # T near INT_MAX: the block count is computed in 64 bits (no overflow)
    big = 2**31 - 1
    assert lib.moe_dispatch_workspace_size(big, 1, 4) == -(-big // 256) * 4 * 4
    ws = lib.moe_expert_compute_workspace_size(2, 128, 256, 128)
    # xq, xs, zq, zs, then the fused GEMM's scratch: a tile ticket and one
    # count per 128-row block (ceil(rows/128) plus one per possible expert),
    # then the per-source layout's slot row of every packed row (int32)
    sync = (1 + 2 + 1024) * 4
    assert ws == 2 * 128 * 256 + 2 * 2 * 128 * 4 + 2 * 128 * 128 + 2 * 1 * 128 * 4 + \
        (sync + 255) // 256 * 256 + 2 * 128 * 4
    assert lib.moe_expert_compute_workspace_size(2, 128, 200, 128) == 0   # H % 128 != 0


@pytest.mark.parametrize("E,R,rows,H,I", [(2, 128, 0, 256, 128), (256, 4096, 0, 7168, 2048),
                                          (128, 2048, 32768, 4096, 1536), (3, 5, 7, 128, 384)])
def test_workspace_layout_is_the_carved_one(lib, E, R, rows, H, I):
    """The workspace offsets the library exports (and api.MoeLayerBuffers'
    views use) are ordered, 256-byte aligned, hold each part's bytes, and end
    at the size the workspace-size query returns."""
    off = (ctypes.c_size_t * 7)()
    assert lib.moe_expert_compute_workspace_layout(E, R, rows, H, I, off) == 0
    xq, xs, zq, zs, sync, sync_bytes, total = list(off)
    n = rows or E * R
    parts = [(xq, n * H), (xs, n * (H // 128) * 4), (zq, n * I), (zs, n * (I // 128) * 4),
             (sync, sync_bytes)]
    for (o, size), (o_next, _) in zip(parts, parts[1:] + [(total, 0)]):
        assert o % 256 == 0 and o + size <= o_next
    assert total == lib.moe_expert_compute_ex_workspace_size(E, R, rows, H, I)
    assert sync_bytes >= lib.moe_gemm_gateup_down_sync_size(E, R, rows)
    assert lib.moe_expert_compute_workspace_layout(E, R, rows, 200, I, off) == -1
    assert lib.moe_expert_compute_workspace_layout(E, R, rows, H, I, None) == -1


def test_gemm_launch_form_query(lib):
    """Forced forms answer without a device; bad sizes and flag bits are
    rejected; MOE_GEMM_MAX_CTAS(n) is a known flag."""
    assert lib.moe_expert_compute_gemm_launches(8, 128, 0, 256, 2) == 1
    assert lib.moe_expert_compute_gemm_launches(8, 128, 0, 256, 4 | (100 << 16)) == 2
    assert lib.moe_expert_compute_gemm_launches(8, 128, 0, 200, 2) == -1
    assert lib.moe_expert_compute_gemm_launches(8, 128, 0, 256, 2 | 4) == -1
    assert lib.moe_expert_compute_gemm_launches(8, 128, 0, 256, 8) == -1


FAKE = ctypes.c_void_p(4096)   # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("case,expected", [
    (dict(H=200), -1),                  # H % 128 != 0
    (dict(K=9), -1),                    # K > E
    (dict(T=-1), -1),
    (dict(E=0), -1),
    (dict(R=0), -1),
    (dict(counts=None), -1),            # null output
    (dict(x=None), -1),                 # null input with T > 0
    (dict(ws_bytes=8), -3),             # workspace too small
    (dict(ws=None), -3),
])
def test_dispatch_rejects_on_host(lib, case, expected):
    a = dict(x=FAKE, idx=FAKE, T=112, H=256, K=2, E=8, R=128, recv=FAKE, counts=FAKE, src=FAKE,
             st=FAKE, ws=FAKE, ws_bytes=1 << 20)
    a.update(case)
    if "K" in case:
        a["E"] = 8
    r = lib.moe_dispatch(a["x"], a["idx"], None, a["T"], a["H"], a["K"], a["E"], a["R"], a["recv"],
                         a["counts"], a["src"], a["st"], a["ws"], a["ws_bytes"], None)
    assert r == expected


def test_compute_and_combine_reject_on_host(lib):
    assert lib.moe_expert_compute(FAKE, FAKE, 2, 128, 256, 100, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, 1 << 30, None) == -1           # I % 128
    assert lib.moe_expert_compute(FAKE, FAKE, 2, 128, 256, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, 16, None) == -3                # workspace too small
    assert lib.moe_expert_compute(FAKE, FAKE, 2, 128, 256, 128, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, 1 << 30, None) == -1           # null weights
    misaligned = ctypes.c_void_p(4096 + 8)
    assert lib.moe_expert_compute(FAKE, FAKE, 2, 128, 256, 128, misaligned, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, FAKE, 1 << 30, None) == -1     # TMA needs 16-byte alignment
    assert lib.moe_combine(None, FAKE, FAKE, 4, 256, 2, 8, 128, FAKE, None) == -1
    assert lib.moe_combine(FAKE, FAKE, FAKE, 4, 256, 40, 8, 128, FAKE, None) == -1   # K > 32
    assert lib.moe_gemm_down(FAKE, FAKE, FAKE, 2, 128, 256, 128, FAKE, FAKE, None, FAKE, None) == -1
    assert lib.moe_quantize_fp8(FAKE, FAKE, 2, 128, 250, FAKE, FAKE, None) == -1


def test_packed_entry_points_reject_on_host(lib):
    """The packed layout's calls validate before launching: the receive buffer
    must have room for every kept route (min(T*K, E*R) rows)."""
    ws = 1 << 20
    # T*K = 224 routes, E*R = 1024 capacity rows -> at least 224 rows
    assert lib.moe_dispatch_packed(FAKE, FAKE, None, 112, 256, 2, 8, 128, 223, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, ws, None) == -1
    assert lib.moe_dispatch_packed(FAKE, FAKE, None, 112, 256, 2, 8, 128, 0, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, ws, None) == -1
    assert lib.moe_dispatch_packed(FAKE, FAKE, None, 112, 256, 2, 8, 128, 224, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, 8, None) == -3          # workspace checked next
    assert lib.moe_dispatch_packed(FAKE, FAKE, None, 112, 200, 2, 8, 128, 224, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, ws, None) == -1         # H % 128
    # packed compute: workspace sized by rows (xq, xs, zq, zs, the GEMM scratch
    # and the slot table, each 256-byte aligned)
    al = lambda v: (v + 255) // 256 * 256
    ws82 = lib.moe_expert_compute_packed_workspace_size(82, 256, 128)
    assert ws82 == al(al(al(al(al(al(82 * 256) + 82 * 2 * 4) + 82 * 128) + 82 * 1 * 4) +
                         (1 + 1 + 1024) * 4) + 82 * 4)
    assert lib.moe_expert_compute_packed_workspace_size(2 * 128, 256, 128) == \
        lib.moe_expert_compute_workspace_size(2, 128, 256, 128)
    assert lib.moe_expert_compute_packed_workspace_size(0, 256, 128) == 0
    assert lib.moe_expert_compute_packed(FAKE, FAKE, 2, 128, 82, 256, 128, FAKE, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, FAKE, ws82 - 1, None) == -3
    assert lib.moe_expert_compute_packed(FAKE, FAKE, 2, 128, 0, 256, 128, FAKE, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, FAKE, ws82, None) == -1
    assert lib.moe_combine_packed(FAKE, 0, FAKE, FAKE, 4, 256, 2, FAKE, None) == -1
    assert lib.moe_combine_packed(FAKE, 82, FAKE, FAKE, 4, 256, 33, FAKE, None) == -1  # K > 32


def test_dispatch_ex_rejects_on_host(lib):
    ws = 1 << 20
    args = lambda bits, rows: (FAKE, FAKE, bits, None, 112, 256, 2, 8, 128, rows, FAKE, FAKE, FAKE,
                               FAKE, FAKE, ws, None)
    assert lib.moe_dispatch_ex(*args(16, 0)) == -1       # ids are int32 or int64
    assert lib.moe_dispatch_ex(*args(8, 0)) == -1
    assert lib.moe_dispatch_ex(*args(32, 100)) == -1     # packed: fewer rows than routes
    assert lib.moe_dispatch_ex(*args(64, -5)) == -1


def test_gemm_gateup_down_sync_size_and_rejections(lib):
    """The fused GEMM launch's scratch: a tile ticket plus one completion count
    per 128-row block, bounded by E*ceil(R/128) (padded) and additionally by
    ceil(rows/128) + E (packed, one partial block per expert)."""
    sz = lib.moe_gemm_gateup_down_sync_size
    assert sz(2, 128, 0) == (1 + 2) * 4
    assert sz(4, 1000, 0) == (1 + 4 * 8) * 4
    assert sz(4, 1000, 300) == (1 + 3 + 4) * 4
    assert sz(256, 4096, 131072) == (1 + 1024 + 256) * 4
    assert sz(0, 128, 0) == 0 and sz(2, 128, -5) == 0
    args = lambda **k: [k.get(n, d) for n, d in (
        ("xq", FAKE), ("xs", FAKE), ("counts", FAKE), ("E", 2), ("R", 128), ("rows", 0),
        ("H", 256), ("I", 128), ("w13", FAKE), ("s13", FAKE), ("w2", FAKE), ("s2", FAKE),
        ("zq", FAKE), ("zs", FAKE), ("out", FAKE), ("st", FAKE), ("sync", FAKE),
        ("sync_bytes", 12), ("flags", 0), ("stream", None))]
    f = lib.moe_gemm_gateup_down
    assert f(*args(sync_bytes=11)) == -3                  # one int short
    assert f(*args(sync=None)) == -3
    assert f(*args(sync=ctypes.c_void_p(4096 + 2))) == -3  # counts are 4-byte words
    assert f(*args(H=200)) == -1
    assert f(*args(flags=8)) == -1                        # unknown flag bit
    assert f(*args(flags=2 | 4)) == -1                    # one launch and two launches at once
    assert f(*args(rows=-1)) == -1
    assert f(*args(out=None)) == -1
    assert f(*args(zq=ctypes.c_void_p(4096 + 8))) == -1   # TMA source must be 16-byte aligned


def test_source_slot_entry_points_reject_on_host(lib):
    """The per-source layout's calls validate before any launch: the BF16 and
    FP8 slot dispatches and the GEMMs on FP8 slots."""
    mis4, mis8 = ctypes.c_void_p(4096 + 4), ctypes.c_void_p(4096 + 8)

    def dq(**k):
        a = dict(x=FAKE, idx=FAKE, bits=64, T=64, H=256, K=2, E=8, L=2, mt=16, off=None, xq=FAKE,
                 xs=FAKE, counts=FAKE, seg=FAKE, src=FAKE, st=FAKE)
        a.update(k)
        return lib.moe_dispatch_quant_source_slots(
            a["x"], a["idx"], a["bits"], None, a["T"], a["H"], a["K"], a["E"], a["L"], a["mt"],
            a["off"], a["xq"], a["xs"], a["counts"], a["seg"], a["src"], a["st"], None)
    assert dq(L=0) == -1
    assert dq(L=3) == -1                       # E % L != 0
    assert dq(mt=0) == -1
    assert dq(bits=16) == -1
    assert dq(H=200) == -1
    assert dq(xq=None) == -1 and dq(xs=None) == -1
    assert dq(xq=mis4) == -1                   # codes are stored 8 bytes at a time
    assert dq(counts=None) == -1 and dq(seg=None) == -1
    assert lib.moe_dispatch_source_slots(FAKE, FAKE, 64, None, 64, 256, 2, 8, 2, 16, None, None,
                                         FAKE, FAKE, FAKE, FAKE, None) == -1   # null recv
    assert lib.moe_dispatch_source_slots(FAKE, FAKE, 64, None, 64, 256, 2, 8, 2, 16, None, mis8,
                                         FAKE, FAKE, FAKE, FAKE, None) == -1   # recv alignment

    ws = lib.moe_expert_compute_workspace_size(8, 4 * 16, 256, 128)
    assert ws > 0

    def gs(**k):
        a = dict(xq=FAKE, xs=FAKE, seg=FAKE, E=8, L=2, mt=16, H=256, I=128, w13=FAKE, s13=FAKE,
                 w2=FAKE, s2=FAKE, out=FAKE, st=FAKE, ws=FAKE, ws_bytes=ws, flags=0)
        a.update(k)
        return lib.moe_gemm_source_slots(
            a["xq"], a["xs"], a["seg"], a["E"], a["L"], a["mt"], a["H"], a["I"], a["w13"],
            a["s13"], a["w2"], a["s2"], a["out"], a["st"], a["ws"], a["ws_bytes"], a["flags"], None)
    assert gs(xq=mis8) == -1                   # TMA reads the packed rows; the slots 16-byte aligned
    assert gs(xq=None) == -1 and gs(xs=None) == -1 and gs(seg=None) == -1
    assert gs(I=100) == -1 and gs(L=3) == -1 and gs(mt=0) == -1
    assert gs(flags=8) == -1
    assert gs(ws_bytes=ws - 1) == -3 and gs(ws=None) == -3
    assert gs(ws=ctypes.c_void_p(4096 + 128)) == -3   # 256-byte aligned workspace


def test_header_compiles_as_c(tmp_path):
    """include/moe.h is plain C: the C layer driver compiles against it with
    gcc in C11 mode, warnings as errors (compile only; it runs in the GPU
    tests)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.isdir(cuda_inc):
        pytest.skip("gcc or the CUDA headers not found")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-c",
                    "-I", os.path.join(root, "include"), "-I", cuda_inc,
                    os.path.join(root, "tests", "capi", "layer_main.c"),
                    "-o", str(tmp_path / "layer_main.o")], check=True)


def test_layer_forward_path_choice_on_host(monkeypatch):
    """MoeLayerBuffers.forward takes the fused dispatch+quant path unless asked
    not to, on every layout, and calls the matching entry points in order (the
    lane is built in host memory and the entry points are recorded, so nothing
    reaches a GPU)."""
    from token_dispatch_grouped_topk_gb300 import api
    names = ["moe_dispatch", "moe_expert_compute", "moe_combine", "moe_dispatch_quant",
             "moe_gemm_gateup_down", "moe_dispatch_packed", "moe_expert_compute_packed",
             "moe_combine_packed", "moe_dispatch_source_slots",
             "moe_expert_compute_source_slots", "moe_dispatch_quant_source_slots",
             "moe_gemm_source_slots"]
    calls = []
    for n in names:
        monkeypatch.setattr(api, n, lambda *a, _n=n, **k: calls.append(_n))
    T, E, K, H, I, L, mt = 8, 4, 2, 128, 128, 2, 4
    cpu = torch.device("cpu")
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    idx = torch.zeros(T, K, dtype=torch.int64)
    w = torch.zeros(T, K)
    lanes = {
        "padded": (api.MoeLayerBuffers(T, E, K, H, I, 8, cpu),
                   ["moe_dispatch_quant", "moe_gemm_gateup_down", "moe_combine"],
                   ["moe_dispatch", "moe_expert_compute", "moe_combine"]),
        "packed": (api.MoeLayerBuffers(T, E, K, H, I, 8, cpu, packed=True),
                   ["moe_dispatch_quant", "moe_gemm_gateup_down", "moe_combine_packed"],
                   ["moe_dispatch_packed", "moe_expert_compute_packed", "moe_combine_packed"]),
        "source_slots": (api.MoeLayerBuffers(T, E, K, H, I, (E // L) * mt, cpu, source_slots=mt,
                                             L=L),
                         ["moe_dispatch_quant_source_slots", "moe_gemm_source_slots",
                          "moe_combine"],
                         ["moe_dispatch_source_slots", "moe_expert_compute_source_slots",
                          "moe_combine"]),
    }
    for name, (lane, fused, separate) in lanes.items():
        for kw, want in (({}, fused), ({"fused": True}, fused), ({"fused": False}, separate)):
            calls.clear()
            lane.forward(x, idx, w, None, None, None, None, **kw)
            assert calls == want, (name, kw, calls)
        calls.clear()
        lane.forward_fused(x, idx, w, None, None, None, None)
        assert calls == fused, name
    # the per-source lane forms its FP8 slots only on the fused path
    lane = lanes["source_slots"][0]
    xq, xs = lane.slots_fp8
    assert xq.shape == (E, (E // L) * mt, H) and xq.dtype == torch.uint8
    assert xs.shape == (E, (E // L) * mt, H // 128) and xs.dtype == torch.float32
