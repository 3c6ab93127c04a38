"""flash_gau_forward_noalloc, the entry point for callers that cannot
allocate device memory (for instance a plugin whose host framework owns the
device memory pool), checked through the C ABI against flash_gau_forward on
the same inputs, on two calls in a row (the second call reuses the static
scratch the first one left behind).  Both run the same kernels in the same
order, so their outputs must agree bit for bit; the output is also held to
the oracle at the layer's tolerance.  Collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from gpu_harness import Case, TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


@pytest.mark.parametrize("shape", [
    # B, T, d, e, s, C, causal, dtype
    (1, 1024, 768, 1536, 128, 256, True, "bf16"),
    (2, 512, 256, 512, 128, 128, False, "bf16"),
    (1, 256, 64, 128, 32, 64, True, "fp32"),
])
def test_noalloc_matches_workspace_entry_point(shape):
    from efficient_attention_transformer_gb300 import binding as bd
    B, T, d, e, s, C, causal, dtype = shape
    case = Case(B, T, d, e, s, C, causal, dtype, seed=77)
    assert case.weights.workspace_bytes(B, T, C, causal) <= bd.NOALLOC_SCRATCH_BYTES
    same = case.run()
    oracle, _ = case.reference()
    for _ in range(2):
        out = torch.full_like(case.X, float("nan"))
        bd.forward_noalloc(case.X, case.weights, C, causal, out=out)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all()
        assert np.array_equal(got, same)
        assert rel_err(got, oracle) <= TOL[dtype]


def test_noalloc_rejects_problems_beyond_the_scratch():
    from efficient_attention_transformer_gb300 import binding as bd
    case = Case(1, 8192, 768, 1536, 128, 256, True, "bf16", seed=78)
    assert case.weights.workspace_bytes(1, 8192, 256, True) > bd.NOALLOC_SCRATCH_BYTES
    L = bd.lib()
    st = L.flash_gau_forward_noalloc(case.X.data_ptr(), ctypes.byref(case.weights.c), 1, 8192,
                                     256, 1, bd.BF16, case.out.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == bd.EWORKSPACE
