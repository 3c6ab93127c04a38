"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs, element by element.

Bar: max|O_gpu - O_oracle| <= tol * max|O_oracle| with tol = 1e-4 for fp32
io and 2e-2 for bf16 io.  Every intermediate the workspace holds (U, V, the
four heads, the chunk states, the prefix states, the gated product) is
checked against the oracle's own intermediate, relative to that tensor's
maximum, because the global term dominates |O| and would hide a broken
local term."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300.synthetic import WORKLOADS
from gpu_harness import Case, TOL, TOL_INTER, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


def _check_all(case, O, ref, inter):
    tol, tol_i = TOL[case.dtype], TOL_INTER[case.dtype]
    errs = {"O": rel_err(O, ref)}
    M = case.B * case.T
    errs["U"] = rel_err(case.intermediate("U"), inter["U"].reshape(M, -1))
    errs["V"] = rel_err(case.intermediate("V"), inter["V"].reshape(M, -1))
    errs["heads"] = rel_err(case.intermediate("heads"), inter["heads"].reshape(4, M, -1))
    # bf16 forms no chunk states or prefixes when the global term is zero for
    # every chunk (causal with a single chunk, or lin_scale 0)
    lin_off = case.dtype == "bf16" and case.local_scale != 0 and (
        case.lin_scale == 0 or (case.causal and case.T == case.C))
    if not lin_off:
        errs["state"] = rel_err(case.intermediate("state"),
                                inter["state"].reshape(-1, case.s, case.e))
    pre = inter["prefix"] * case.lin_scale
    if not case.causal:
        pre = pre[:, 0]
    pre = pre.reshape(-1, case.s, case.e)
    if case.lin_scale != 0 and not lin_off:
        errs["prefix"] = rel_err(case.intermediate("prefix"), pre)
    errs["gated"] = rel_err(case.intermediate("gated"), inter["gated"].reshape(M, -1))
    print(case.dtype, {k: "%.2e" % v for k, v in errs.items()})
    assert errs["O"] <= tol, errs
    for k, v in errs.items():
        if k != "O":
            assert v <= tol_i, (k, errs)
    assert case.status() == 0


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_matches_oracle(name):
    w = WORKLOADS[name]
    case = Case(**w)
    O = case.run()
    ref, inter = case.reference()
    _check_all(case, O, ref, inter)


@pytest.mark.parametrize("name", ["tiny_causal_fp32_T256", "lm112m_causal_B8_T1024",
                                  "mlm112m_noncausal_B32_T512", "wide500m_causal_T8192_C512"])
def test_local_term_alone(name):
    """lin_scale = 0 (the LocalOnly ablation): the gated product is U times
    the chunk-local relu^2 term only, so the local path is checked on its
    own scale."""
    w = dict(WORKLOADS[name])
    if w["dtype"] == "bf16":
        w.update(B=1, T=min(w["T"], 2048))
    case = Case(**w, lin_scale=0.0)
    O = case.run()
    ref, inter = case.reference()
    _check_all(case, O, ref, inter)


EDGE = [
    # name, B, T, d, e, s, C, causal, dtype
    ("fp32_ragged_tiles", 3, 96, 40, 72, 24, 48, False, "fp32"),
    ("fp32_ragged_tiles_causal", 3, 96, 40, 72, 24, 48, True, "fp32"),
    ("fp32_single_token_chunks", 2, 8, 16, 16, 8, 1, True, "fp32"),
    ("fp32_one_chunk_quad", 2, 160, 32, 64, 16, 160, True, "fp32"),
    ("bf16_one_chunk_causal", 1, 256, 128, 256, 128, 256, True, "bf16"),
    ("bf16_one_chunk_noncausal", 1, 256, 128, 256, 128, 256, False, "bf16"),
    ("bf16_single_tile", 3, 128, 128, 256, 128, 128, True, "bf16"),
    ("bf16_many_chunks_noncausal", 2, 2048, 384, 512, 128, 128, False, "bf16"),
    ("bf16_c1024_causal", 1, 2048, 256, 512, 128, 1024, True, "bf16"),
    ("bf16_max_chunk", 1, 4096, 128, 256, 128, 4096, True, "bf16"),
]


@pytest.mark.parametrize("name,B,T,d,e,s,C,causal,dtype", EDGE, ids=[x[0] for x in EDGE])
def test_edge_shapes(name, B, T, d, e, s, C, causal, dtype):
    case = Case(B, T, d, e, s, C, causal, dtype, seed=101)
    O = case.run()
    ref, inter = case.reference()
    _check_all(case, O, ref, inter)


def test_repeat_calls_are_bitwise_identical_and_stream_aware():
    case = Case(**WORKLOADS["lm112m_causal_B8_T1024"])
    a = case.run().copy()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        from efficient_attention_transformer_gb300 import binding as bd
        out2 = torch.empty_like(case.X)
        bd.forward(case.X, case.weights, case.C, case.causal, out=out2,
                   workspace=case.workspace, stream=s)
    s.synchronize()
    np.testing.assert_array_equal(out2.double().cpu().numpy(), a)


def test_wrong_device_arch_is_not_reported_and_status_clear():
    from efficient_attention_transformer_gb300 import binding as bd
    case = Case(**WORKLOADS["tiny_causal_fp32_T256"])
    case.run()
    assert bd.workspace_status(case.workspace) == 0
