"""GPU parity of the flash_block wrapper (pre-norm, RoPE on the four heads at
global positions, residual) through flash_gau_block_forward, against the
oracle's flash_block on the same seeded inputs.

The residual adds X, whose magnitude would hide errors in the layer's
output, so Y - X is compared (relative to its own maximum) with the same
bar as the layer alone: 1e-4 for fp32 io, 2e-2 for bf16 io.  The normalised
input and the rotated heads are checked as intermediates."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from efficient_attention_transformer_gb300.synthetic import WORKLOADS
from gpu_harness import Case, TOL, TOL_INTER, rel_err
from oracle import flash_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


def _norm_params(d, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "layer":
        return rng.normal(1.0, 0.1, d), rng.normal(0.0, 0.1, d)
    return np.array([float(np.sqrt(d)) * rng.uniform(0.8, 1.2)]), None


def _run_block(case, kind, pos_offset, base=10000.0):
    g, b = _norm_params(case.d, kind, 123)
    dev = case.X.device
    g_t = torch.tensor(g, dtype=torch.float32, device=dev)
    b_t = torch.tensor(b, dtype=torch.float32, device=dev) if b is not None else None
    out = torch.empty_like(case.X)
    bd.block_forward(case.X, case.weights, case.C, case.causal,
                     norm=bd.NORM_LAYER if kind == "layer" else bd.NORM_SCALE,
                     norm_g=g_t, norm_b=b_t, norm_eps=1e-5, rope=True, rope_base=base,
                     pos_offset=pos_offset, residual=True, out=out, workspace=case.workspace)
    torch.cuda.synchronize()
    i = case.inp
    ref, inter = flash_block(i["X"], i["W_u"], i["W_v"], i["W_z"], i["W_o"], i["gamma"],
                             i["beta"], i["relpos"], case.C, case.causal, case.lin_scale,
                             norm=kind, norm_g=g if kind == "layer" else g[0], norm_b=b,
                             norm_eps=1e-5, rope_on=True, rope_base=base,
                             pos_offset=pos_offset)
    return out.double().cpu().numpy(), ref, inter


def _xn(case):
    tdt = case.X.dtype
    n = case.B * case.T * case.d
    raw = case.workspace[case.layout["xn"]:]
    t = raw[: n * (2 if tdt == torch.bfloat16 else 4)].view(tdt).view(case.B, case.T, case.d)
    return t.double().cpu().numpy()


CASES = [
    # name, workload overrides, norm, pos_offset
    ("fp32_tiny_layer", dict(WORKLOADS["tiny_causal_fp32_T256"]), "layer", 0),
    ("fp32_tiny_scale_offset", dict(WORKLOADS["tiny_causal_fp32_T256"]), "scale", 37),
    ("fp32_noncausal_layer", dict(B=2, T=128, d=48, e=96, s=16, C=32, causal=False,
                                  dtype="fp32", seed=21), "layer", 5),
    ("bf16_lm_layer", dict(WORKLOADS["lm112m_causal_B8_T1024"]), "layer", 0),
    ("bf16_mlm_scale", dict(WORKLOADS["mlm112m_noncausal_B32_T512"]), "scale", 0),
    ("bf16_long_layer_offset", dict(WORKLOADS["long_causal_B2_T8192"]), "layer", 4096),
    ("bf16_c512_layer", dict(WORKLOADS["wide500m_causal_T8192_C512"]), "layer", 0),
]


@pytest.mark.parametrize("name,w,kind,pos_offset", CASES, ids=[c[0] for c in CASES])
def test_block_matches_oracle(name, w, kind, pos_offset):
    # the listing's normalisation of the global term (1/C) keeps it from
    # dominating the output
    case = Case(**w, lin_scale=1.0 / w["C"])
    Y, ref, inter = _run_block(case, kind, pos_offset)
    X = case.inp["X"].astype(np.float64)
    tol, tol_i = TOL[case.dtype], TOL_INTER[case.dtype]
    errs = {"Y-X": rel_err(Y - X, ref - X),
            "xn": rel_err(_xn(case), inter["Xn"]),
            "heads": rel_err(case.intermediate("heads"),
                             inter["heads"].reshape(4, case.B * case.T, -1)),
            "gated": rel_err(case.intermediate("gated"),
                             inter["gated"].reshape(case.B * case.T, -1))}
    print(name, {k: "%.2e" % v for k, v in errs.items()})
    assert errs["Y-X"] <= tol, errs
    for k in ("xn", "heads", "gated"):
        assert errs[k] <= tol_i, (k, errs)
    assert case.status() == 0


def test_block_without_options_is_the_layer():
    """norm NONE, no RoPE, no residual: bitwise the same as flash_gau_forward."""
    case = Case(**WORKLOADS["lm112m_causal_B8_T1024"])
    a = case.run().copy()
    out = torch.empty_like(case.X)
    bd.block_forward(case.X, case.weights, case.C, case.causal, norm=bd.NORM_NONE,
                     rope=False, residual=False, out=out, workspace=case.workspace)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.double().cpu().numpy(), a)
