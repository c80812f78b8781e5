"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory (runtimes that reserve all device memory at start-up,
hosts that give the library no allocator, loops that cannot pay cudaMalloc's
implicit synchronisation): called through the C ABI,
it must give exactly what moe_dispatch gives with a caller-provided workspace,
on two calls in a row that share its built-in scratch array.  This file is
named so pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

from token_dispatch_grouped_topk_gb300 import _lib, api
from token_dispatch_grouped_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, x, idx, w, E, R):
    T, H = x.shape
    K = idx.shape[1]
    recv = torch.full((E, R, H), -7.0, dtype=torch.bfloat16, device=DEV)
    counts = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    src_map = torch.full((T, K), -5, dtype=torch.int32, device=DEV)
    st = torch.full((2,), 123, dtype=torch.int32, device=DEV)
    rc = lib.moe_dispatch_noalloc(_p(x), _p(idx), _p(w), T, H, K, E, R, _p(recv), _p(counts),
                                  _p(src_map), _p(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, _lib.STATUS.get(rc, rc)
    return recv, counts, src_map, st


def _same(a, b, x):
    recv_a, counts_a, map_a, st_a = a
    recv_b, counts_b, map_b, st_b = b
    assert torch.equal(counts_a, counts_b)
    assert torch.equal(map_a, map_b)
    assert torch.equal(st_a, st_b)
    keep = map_a.view(-1) >= 0
    rows = map_a.view(-1)[keep].long()
    H = x.shape[1]
    assert torch.equal(recv_a.view(-1, H)[rows].view(torch.int16), recv_b.view(-1, H)[rows].view(torch.int16))


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.load()
    # call 1: skewed random routing with capacity drops and an invalid id
    g = torch.Generator().manual_seed(77)
    T, E, K, R, H = 1000, 64, 8, 96, 512
    idx = torch.randint(-1, E, (T, K), generator=g)
    idx[:, 0] = torch.randint(0, 4, (T,), generator=g)          # four hot experts overflow R
    idx[9, 3] = E + 1
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    idx, w = idx.to(DEV), torch.rand(T, K, generator=g).to(DEV)
    ref = api.moe_dispatch(x, idx, w, E, R)
    got = _noalloc(lib, x, idx, w, E, R)
    torch.cuda.synchronize()
    _same(got, ref, x)
    st = got[3].cpu().tolist()
    assert st[0] & api.DEV_CAPACITY_DROPPED and st[0] & api.DEV_BAD_EXPERT_ID and st[1] > 0
    # call 2, right after: the traced scenario, different sizes, same scratch array
    d = W.make_layer_inputs("traced", seed=3, device=DEV, weights=False)
    wl = d["wl"]
    ref2 = api.moe_dispatch(d["x"], d["topk_idx"], d["topk_w"], wl.E, wl.R)
    got2 = _noalloc(lib, d["x"], d["topk_idx"], d["topk_w"], wl.E, wl.R)
    torch.cuda.synchronize()
    _same(got2, ref2, d["x"])
    assert got2[1].cpu().tolist() == [111, 1, 0, 0, 0, 0, 1, 111]


def test_noalloc_dispatch_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.load()
    # E * ceil(T / 32) int32 = 1024 * 2048 * 4 bytes = 8 MiB > 1 MiB
    T, K, E = 65536, 8, 1024
    assert lib.moe_dispatch_workspace_size(T, K, E) > (1 << 20)
    # Null pointers throughout: the size check must answer first; were it
    # missing, the dispatch would reject the null pointers on the host and
    # still launch nothing.
    rc = lib.moe_dispatch_noalloc(None, None, None, T, 256, K, E, 16, None, None, None, None, None)
    assert rc == -3
