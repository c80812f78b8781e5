"""The C ABI driven from a plain C program: tests/capi/layer_main.c has no
Python or PyTorch in its process, only the CUDA runtime for memory and a
stream.  It is compiled here with gcc against include/moe.h and the library,
runs one layer on arrays written to files (the separate path, or the default
fused path: moe_dispatch_quant, moe_gemm_gateup_down, moe_combine), and its y,
counts, source map and status must equal the same layer run through the
Python binding."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from token_dispatch_grouped_topk_gb300 import _lib, api
from token_dispatch_grouped_topk_gb300 import build as B
from token_dispatch_grouped_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"


@pytest.fixture(scope="module")
def layer_main(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    _lib.load()
    exe = str(tmp_path_factory.mktemp("capi") / "layer_main")
    subprocess.run([gcc, "-O2", "-std=c11", "-Wall", "-I", os.path.join(ROOT, "include"),
                    "-I", f"{CUDA}/include", os.path.join(ROOT, "tests", "capi", "layer_main.c"),
                    "-o", exe, "-L", B.BUILD_DIR, "-lmoe_gb300", "-L", f"{CUDA}/lib64", "-lcudart",
                    f"-Wl,-rpath,{B.BUILD_DIR}", f"-Wl,-rpath,{CUDA}/lib64"], check=True)
    return exe


def _raw(t):
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float8_e4m3fn):
        t = t.view(torch.uint8 if t.dtype == torch.float8_e4m3fn else torch.int16)
    return t.numpy()


@pytest.mark.parametrize("path", ["separate", "fused"])
@pytest.mark.parametrize("case", ["traced", "ragged"])
def test_c_program_layer_matches_python_binding(layer_main, tmp_path, case, path):
    if case == "traced":
        d = W.make_layer_inputs("traced", seed=9, device="cpu")
        wl = d["wl"]
        T, H, K, E, R, I = wl.T, wl.H, wl.K, wl.E, wl.R, wl.I
        x, idx, w = d["x"], d["topk_idx"], d["topk_w"]
        w13, s13, w2, s2 = d["w13"], d["s13"], d["w2"], d["s2"]
    else:
        # several tiles per expert, a ragged tail, capacity drops and a padding route
        T, H, K, E, R, I = 600, 512, 4, 12, 160, 256
        x = W.activations(T, H, 10, "cpu")
        idx, w = W.router(T, E, K, torch.zeros(E), 11, "cpu")
        idx[7, 2] = -1
        w13, s13, w2, s2 = W.expert_weights(E, H, I, 12, "cpu")
    for name, t in (("x", x), ("idx", idx), ("w", w), ("w13", w13), ("s13", s13), ("w2", w2),
                    ("s2", s2)):
        _raw(t).tofile(str(tmp_path / f"{name}.bin"))
    argv = [layer_main, str(tmp_path), str(T), str(H), str(K), str(E), str(R), str(I)]
    run = subprocess.run(argv + (["fused"] if path == "fused" else []), capture_output=True,
                         text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    y_c = np.fromfile(str(tmp_path / "y.bin"), dtype=np.int16).reshape(T, H)
    counts_c = np.fromfile(str(tmp_path / "counts.bin"), dtype=np.int32)
    src_c = np.fromfile(str(tmp_path / "src_map.bin"), dtype=np.int32).reshape(T, K)
    st_c = np.fromfile(str(tmp_path / "status.bin"), dtype=np.int32)

    dev = torch.device("cuda")
    buf = api.MoeLayerBuffers(T, E, K, H, I, R, dev)
    y = buf.forward(x.to(dev), idx.to(dev), w.to(dev), w13.to(dev), s13.to(dev), w2.to(dev),
                    s2.to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(counts_c, buf.counts.cpu().numpy())
    assert np.array_equal(src_c, buf.src_map.cpu().numpy())
    assert np.array_equal(st_c, buf.dev_status.cpu().numpy())
    assert np.array_equal(y_c, y.cpu().view(torch.int16).numpy())
    assert int(st_c[0]) & api.DEV_TIMEOUT == 0
    if case == "ragged":
        assert int(st_c[1]) > 0          # the capacity of 160 rows drops routes
