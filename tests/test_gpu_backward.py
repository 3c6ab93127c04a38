"""GPU parity of the backward pass (flash_gau_backward) against the float64
oracle's chain-rule gradients (oracle.flash_gau_backward, itself pinned by
finite differences), on the same seeded inputs.

Both sides see the same io-typed inputs (bf16-rounded for bf16 io).  For
fp32 io the GPU computes in fp32 throughout: every gradient gets 1e-4 of its
maximum.  For bf16 io the large contractions run on the tensor cores with
bf16 operands (the gated product and dPre rounded to bf16, 2^-9 each), so
every gradient gets 1e-2, the bar of the layer's own bf16 intermediates."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from efficient_attention_transformer_gb300.synthetic import make_inputs
from gpu_harness import rel_err, torch_dtype
from oracle import flash_gau_backward

pytestmark = pytest.mark.gpu

TOL_W = {"fp32": 1e-4, "bf16": 1e-2}
TOL_X = {"fp32": 1e-4, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


def _run(B, T, d, e, s, C, causal, dtype, lin_scale, seed, local_scale=1.0):
    inp = make_inputs(B, T, d, e, s, C, dtype, seed)
    tdt = torch_dtype(dtype)
    dev = torch.device("cuda")
    dO = torch.tensor(np.random.default_rng(seed + 1).normal(size=(B, T, d)), dtype=tdt,
                      device=dev)
    dO64 = dO.double().cpu().numpy()  # the io-typed values both sides use
    W_uvz = np.concatenate([inp["W_u"], inp["W_v"], inp["W_z"]], axis=1)
    w = bd.GauWeights(torch.tensor(W_uvz, dtype=tdt, device=dev),
                      torch.tensor(inp["W_o"], dtype=tdt, device=dev),
                      torch.tensor(inp["gamma"], dtype=torch.float32, device=dev),
                      torch.tensor(inp["beta"], dtype=torch.float32, device=dev),
                      torch.tensor(inp["relpos"], dtype=torch.float32, device=dev),
                      d, e, s, lin_scale, local_scale)
    X = torch.tensor(inp["X"], dtype=tdt, device=dev)
    got = bd.backward(X, dO, w, C, causal)
    torch.cuda.synchronize()
    ref = flash_gau_backward(inp["X"], inp["W_u"], inp["W_v"], inp["W_z"], inp["W_o"],
                             inp["gamma"], inp["beta"], inp["relpos"], C, causal, dO64,
                             lin_scale, local_scale)
    g = {k: v.double().cpu().numpy() for k, v in got.items()}
    errs = {
        "dX": rel_err(g["dX"], ref["dX"].reshape(B, T, d)),
        "dW_uvz": rel_err(g["dW_uvz"], np.concatenate([ref["dW_u"], ref["dW_v"], ref["dW_z"]],
                                                      axis=1)),
        "dW_o": rel_err(g["dW_o"], ref["dW_o"]),
        "dgamma": rel_err(g["dgamma"], ref["dgamma"]),
        "dbeta": rel_err(g["dbeta"], ref["dbeta"]),
        "drelpos": rel_err(g["drelpos"], ref["drelpos"]),
    }
    return errs


@pytest.mark.parametrize("shape,causal,dtype,lin_scale", [
    ((1, 256, 64, 128, 32, 64), True, "fp32", 1.0),
    ((2, 256, 64, 128, 32, 64), False, "fp32", 0.25),
    ((2, 512, 128, 256, 128, 128), True, "bf16", 1.0 / 128),
    ((1, 1024, 256, 512, 128, 256), True, "bf16", 1.0),
    ((2, 512, 128, 384, 64, 128), False, "bf16", 0.5),
    ((1, 384, 96, 160, 64, 128), False, "bf16", 1.0),
    ((1, 256, 64, 128, 32, 256), True, "fp32", 0.0),
    # chunk-level contractions on the tensor cores: value width with a
    # 128-column tile tail, several chunks non-causal
    ((2, 512, 128, 384, 128, 128), True, "bf16", 1.0),
    ((1, 1024, 256, 512, 128, 256), False, "bf16", 1.0 / 256),
    # the layer's full widths (d = 768, e = 1536): the weight gradients run
    # split-K over 36 and 78 output tiles, and the persistent contractions
    # take several rounds of tiles
    ((1, 2048, 768, 1536, 128, 256), True, "bf16", 1.0),
    ((2, 1024, 768, 1536, 128, 256), False, "bf16", 1.0),
    # 40 row pairs of 256: the dA (gate gradient) and dX pair GEMMs run a
    # last partial round of their tiles as 128-column tiles
    ((5, 2048, 512, 512, 128, 256), True, "bf16", 1.0),
])
def test_backward_matches_oracle(shape, causal, dtype, lin_scale):
    B, T, d, e, s, C = shape
    errs = _run(B, T, d, e, s, C, causal, dtype, lin_scale, seed=61 + T)
    print(dtype, causal, {k: "%.2e" % v for k, v in errs.items()})
    assert errs["dX"] <= TOL_X[dtype], errs
    for k in ("dW_uvz", "dW_o", "dgamma", "dbeta", "drelpos"):
        assert errs[k] <= TOL_W[dtype], (k, errs)


def test_backward_rejects_bad_arguments():
    L = bd.lib()
    dev = torch.device("cuda")
    w = bd.GauWeights(torch.zeros(64, 288, device=dev), torch.zeros(128, 64, device=dev),
                      torch.zeros(4, 32, device=dev), torch.zeros(4, 32, device=dev),
                      torch.zeros(127, device=dev), 64, 128, 32)
    import ctypes
    assert L.flash_gau_backward_workspace_bytes(1, 100, 64, ctypes.byref(w.c), 1, bd.FP32) == 0
    g = bd.Grads()
    X = torch.zeros(1, 128, 64, device=dev)
    st = L.flash_gau_backward(X.data_ptr(), X.data_ptr(), ctypes.byref(w.c), 1, 128, 64, 1,
                              bd.FP32, ctypes.byref(g), X.data_ptr(), 0,
                              torch.cuda.current_stream().cuda_stream)
    assert st == bd.EINVAL  # null gradient pointers


@pytest.mark.parametrize("shape,causal,dtype,local_scale", [
    ((1, 256, 64, 128, 32, 64), True, "fp32", 0.0),       # GlobalOnly
    ((2, 256, 64, 128, 32, 64), False, "fp32", -0.5),
    ((2, 512, 128, 256, 128, 128), True, "bf16", 0.0),
    ((1, 512, 128, 256, 128, 256), False, "bf16", 2.0),
])
def test_backward_with_scaled_local_term(shape, causal, dtype, local_scale):
    """The local term times local_scale (0: the GlobalOnly ablation, whose
    relpos gradient is then exactly zero)."""
    B, T, d, e, s, C = shape
    errs = _run(B, T, d, e, s, C, causal, dtype, 1.0, seed=71 + T, local_scale=local_scale)
    print(dtype, causal, local_scale, {k: "%.2e" % v for k, v in errs.items()})
    for k, v in errs.items():
        assert v <= (TOL_X if k == "dX" else TOL_W)[dtype], (k, errs)
