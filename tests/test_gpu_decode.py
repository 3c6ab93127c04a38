"""GPU parity of the autoregressive decode step (flash_gau_decode_step).

By causality, the output of token t of a sequence is row t of the causal
forward over its first t + 1 tokens: each step is checked against the
oracle's forward on the same seeded inputs (the tokens after t zero-padded
to a multiple of C), across chunk boundaries (the linear cache must then
carry the completed chunks), with the layer's tolerances (1e-4 of the
maximum for fp32 io, 2e-2 for bf16 io)."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from efficient_attention_transformer_gb300.synthetic import make_inputs
from gpu_harness import TOL, rel_err, torch_dtype
from oracle import flash_gau

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


@pytest.mark.parametrize("B,steps,d,e,s,C,dtype,lin_scale,local_scale", [
    (3, 40, 64, 128, 32, 16, "fp32", 1.0, 1.0),
    (2, 70, 96, 160, 64, 32, "fp32", 0.5, 1.0),
    (4, 300, 768, 1536, 128, 256, "bf16", 1.0 / 256, 1.0),
    (17, 20, 128, 256, 128, 8, "bf16", 1.0, 1.0),
    (2, 50, 64, 128, 32, 16, "fp32", 1.0, 0.0),    # GlobalOnly
    (3, 40, 128, 256, 128, 16, "bf16", 1.0, 0.5),
    # the layer's widths with a batch of 64 sequences: the projections run
    # as tensor-core products over 64 (and 1) padded sequence rows
    (64, 260, 768, 1536, 128, 256, "bf16", 1.0 / 256, 1.0),
    (1, 40, 768, 1536, 128, 16, "bf16", 1.0, 1.0),
    # more attention blocks than two an SM in fp32: the one-accumulator form
    (32, 20, 256, 1536, 64, 16, "fp32", 1.0, 1.0),
])
def test_decode_matches_causal_forward(B, steps, d, e, s, C, dtype, lin_scale, local_scale):
    T = -(-steps // C) * C
    inp = make_inputs(B, T, d, e, s, C, dtype, 90 + C)
    X = inp["X"].copy()
    X[:, steps:] = 0.0
    ref, _ = flash_gau(X, inp["W_u"], inp["W_v"], inp["W_z"], inp["W_o"], inp["gamma"],
                       inp["beta"], inp["relpos"], C, True, lin_scale,
                       local_scale=local_scale)
    tdt = torch_dtype(dtype)
    dev = torch.device("cuda")
    W_uvz = np.concatenate([inp["W_u"], inp["W_v"], inp["W_z"]], axis=1)
    w = bd.GauWeights(torch.tensor(W_uvz, dtype=tdt, device=dev),
                      torch.tensor(inp["W_o"], dtype=tdt, device=dev),
                      torch.tensor(inp["gamma"], dtype=torch.float32, device=dev),
                      torch.tensor(inp["beta"], dtype=torch.float32, device=dev),
                      torch.tensor(inp["relpos"], dtype=torch.float32, device=dev),
                      d, e, s, lin_scale, local_scale)
    dec = bd.Decoder(w, B, C)
    Xd = torch.tensor(X, dtype=tdt, device=dev)
    outs = [dec.step(Xd[:, t].contiguous()).double().cpu().numpy() for t in range(steps)]
    torch.cuda.synchronize()
    got = np.stack(outs, axis=1)  # [B, steps, d]
    err = rel_err(got, ref[:, :steps])
    worst = max(rel_err(got[:, t], ref[:, t]) for t in range(steps))
    print(dtype, C, "all %.2e worst step %.2e" % (err, worst))
    assert err <= TOL[dtype], err
    # every step on its own, so that the small outputs of the early tokens
    # are not hidden by the large ones of later tokens
    assert worst <= 2 * TOL[dtype], worst


def test_decode_reset_restarts_the_sequences():
    B, d, e, s, C = 2, 64, 128, 32, 8
    inp = make_inputs(B, C, d, e, s, C, "fp32", 5)
    dev = torch.device("cuda")
    W_uvz = np.concatenate([inp["W_u"], inp["W_v"], inp["W_z"]], axis=1)
    t = lambda a: torch.tensor(a, dtype=torch.float32, device=dev)  # noqa: E731
    w = bd.GauWeights(t(W_uvz), t(inp["W_o"]), t(inp["gamma"]), t(inp["beta"]),
                      t(inp["relpos"]), d, e, s)
    dec = bd.Decoder(w, B, C)
    X = t(inp["X"])
    first = [dec.step(X[:, i].contiguous()).clone() for i in range(C)]
    dec.reset()
    again = [dec.step(X[:, i].contiguous()).clone() for i in range(C)]
    for a, b in zip(first, again):
        assert torch.equal(a, b)
