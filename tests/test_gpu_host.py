"""flash_gau_forward_host: the forward on host buffers, its batch cut into
parts whose copies overlap the layer.  Each batch row is an independent
problem, so the result must equal the device-buffer forward bit for bit (and
the oracle within the layer's tolerance), whatever the number of parts."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from gpu_harness import Case, TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


@pytest.mark.parametrize("shape,causal,dtype", [
    ((2, 1024, 256, 512, 128, 256), True, "bf16"),    # two parts
    ((5, 512, 128, 256, 128, 128), False, "bf16"),    # four parts, the last one row
    ((3, 96, 40, 72, 24, 32), True, "fp32"),          # three parts, ragged widths
    ((1, 256, 64, 128, 32, 64), False, "fp32"),       # one part
])
def test_host_forward_equals_device_forward(shape, causal, dtype):
    B, T, d, e, s, C = shape
    case = Case(B, T, d, e, s, C, causal, dtype, seed=131 + B)
    ref_dev = case.run()
    Xh = case.X.cpu().pin_memory()
    out = bd.forward_host(Xh, case.weights, C, causal)
    torch.cuda.synchronize()
    got = out.double().numpy()
    assert np.array_equal(got, ref_dev)
    ref, _ = case.reference()
    assert rel_err(got, ref) <= TOL[dtype]


def test_host_forward_with_pageable_buffers_and_repeated_calls():
    B, T, d, e, s, C = 2, 512, 128, 256, 128, 128
    case = Case(B, T, d, e, s, C, True, "bf16", seed=140)
    ref_dev = case.run()
    Xh = case.X.cpu()  # pageable
    out = torch.empty_like(Xh)
    for _ in range(3):
        out.zero_()
        bd.forward_host(Xh, case.weights, C, True, out=out)
        torch.cuda.synchronize()
        assert np.array_equal(out.double().numpy(), ref_dev)


def test_host_forward_workspace_checks():
    case = Case(2, 256, 64, 128, 32, 64, True, "fp32", seed=141)
    import ctypes
    L = bd.lib()
    n = L.flash_gau_forward_host_workspace_bytes(2, 256, 64, ctypes.byref(case.weights.c), 1,
                                                 bd.FP32)
    assert n > 2 * 2 * 256 * 64 * 4
    small = torch.zeros(n - 256, dtype=torch.uint8, device="cuda")
    Xh = case.X.cpu()
    out = torch.empty_like(Xh)
    st = L.flash_gau_forward_host(Xh.data_ptr(), ctypes.byref(case.weights.c), 2, 256, 64, 1,
                                  bd.FP32, out.data_ptr(), small.data_ptr(), n - 256,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == bd.EWORKSPACE
    assert L.flash_gau_forward_host_workspace_bytes(2, 250, 64, ctypes.byref(case.weights.c), 1,
                                                    bd.FP32) == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_forward_replays_as_a_cuda_graph(dtype):
    """The forward enqueues only kernels (tensor maps are built on the host
    at capture), so it can be captured once and replayed; a replay on new
    input data equals the eager call bit for bit."""
    B, T, d, e, s, C = (2, 512, 128, 256, 128, 128) if dtype == "bf16" else (1, 192, 64, 96, 32, 64)
    case = Case(B, T, d, e, s, C, True, dtype, seed=161)
    ws, out = case.workspace, case.out
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):  # warm-up outside the capture
        bd.forward(case.X, case.weights, C, True, out=out, workspace=ws, stream=cap)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        bd.forward(case.X, case.weights, C, True, out=out, workspace=ws, stream=cap)
    torch.cuda.synchronize()
    for seed in (1, 2):
        torch.manual_seed(seed)
        case.X.copy_(torch.randn_like(case.X) * (1 + seed))
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        eager = bd.forward(case.X, case.weights, C, True, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got, eager)
