"""Failure handling on the GPU without a GPU fault: bad inputs are reported
through the device status word or rejected on the host, and a device-side
wait that runs out returns MOE_DEV_TIMEOUT with the context still usable."""
import ctypes

import pytest
import torch

from token_dispatch_grouped_topk_gb300 import _lib, api
from token_dispatch_grouped_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bounded_wait_times_out_and_context_survives():
    lib = _lib.load()
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    rc = lib.moe_selftest_bounded_wait(ctypes.c_void_p(st.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert st[0].item() & api.DEV_TIMEOUT
    assert st[1].item() == 3          # both the mbarrier wait and the counter wait gave up
    # the context is still usable: a full layer runs and reports no timeout
    d = W.make_layer_inputs("traced", seed=0, device=DEV)
    wl = d["wl"]
    buf = api.MoeLayerBuffers(wl.T, wl.E, wl.K, wl.H, wl.I, wl.R, torch.device(DEV))
    buf.forward(d["x"], d["topk_idx"], d["topk_w"], d["w13"], d["s13"], d["w2"], d["s2"])
    torch.cuda.synchronize()
    assert buf.dev_status.cpu().tolist() == [0, 0]


def test_bad_expert_ids_are_reported_not_faulted():
    x = torch.randn(64, 256, device=DEV).to(torch.bfloat16)
    idx = torch.randint(0, 8, (64, 2), device=DEV)
    idx[5, 1] = 1 << 40          # far out of range
    idx[6, 0] = -7
    _, counts, src_map, st = api.moe_dispatch(x, idx, None, 8, 32)
    torch.cuda.synchronize()
    assert st[0].item() & api.DEV_BAD_EXPERT_ID
    assert src_map[5, 1].item() == -1 and src_map[6, 0].item() == -1
    assert int(counts.sum()) == 64 * 2 - 2


def test_host_rejections_launch_nothing():
    x = torch.randn(8, 200, device=DEV).to(torch.bfloat16)      # H % 128 != 0
    idx = torch.zeros(8, 2, dtype=torch.int64, device=DEV)
    with pytest.raises(api.MoeError) as ei:
        api.moe_dispatch(x, idx, None, 8, 32)
    assert ei.value.status == -1
    x = torch.randn(8, 256, device=DEV).to(torch.bfloat16)
    with pytest.raises(api.MoeError) as ei:
        api.moe_dispatch(x, idx, None, 8, 32, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert ei.value.status == -3
    torch.cuda.synchronize()
