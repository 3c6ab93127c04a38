"""GPU parity of the variants of the layer's building blocks.

RoPE construction of the relative position bias ("Transformer Quality in
Linear Time", appendix D, Code 4, the branch for windows of 512 positions
and more): flash_gau_rope_toeplitz_bias writes the layer's 2C-1 table from
two learned vectors; it is checked against the oracle's n x n construction
read back into table form, and then fed to the layer, whose output is
checked against the oracle's layer with the oracle's bias."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from efficient_attention_transformer_gb300.synthetic import make_inputs
from gpu_harness import Case, TOL, rel_err
from oracle import rope_toeplitz_bias, toeplitz_relpos

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


def _ab(m, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(0.0, 1.0 / np.sqrt(m), m), rng.normal(0.0, 1.0 / np.sqrt(m), m)


@pytest.mark.parametrize("m,C,base", [(128, 512, 10000.0), (128, 2048, 10000.0),
                                      (64, 1000, 500.0), (2, 7, 10000.0)])
def test_rope_toeplitz_table_matches_oracle(m, C, base):
    a, b = _ab(m, 31 + C)
    want = toeplitz_relpos(rope_toeplitz_bias(a, b, C, base))
    dev = torch.device("cuda")
    got = bd.rope_toeplitz_bias(torch.tensor(a, dtype=torch.float32, device=dev),
                                torch.tensor(b, dtype=torch.float32, device=dev), C, base)
    torch.cuda.synchronize()
    got = got.double().cpu().numpy()
    # fp32 inputs (rounded on the way in) and fp32 sums over m/2 pairs
    assert rel_err(got, want) <= 2e-5, rel_err(got, want)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_layer_with_rope_toeplitz_bias(dtype):
    """C = 512, the window size from which the listing switches to this
    construction: the layer fed with the kernel's table against the oracle's
    layer fed with the oracle's table."""
    B, T, d, e, s, C = 1, 1024, 256, 512, 128, 512
    inp = make_inputs(B, T, d, e, s, C, dtype, 41)
    a, b = _ab(128, 42)
    # scaled so that the bias matters next to the 1/C-scaled scores
    a, b = 4.0 * a, 4.0 * b
    inp["relpos"] = toeplitz_relpos(rope_toeplitz_bias(a, b, C))
    case = Case(B, T, d, e, s, C, True, dtype, seed=41, inputs=inp)
    dev = case.X.device
    bd.rope_toeplitz_bias(torch.tensor(a, dtype=torch.float32, device=dev),
                          torch.tensor(b, dtype=torch.float32, device=dev), C,
                          out=case.weights.relpos)
    O = case.run()
    ref, _ = case.reference()
    assert rel_err(O, ref) <= TOL[dtype], rel_err(O, ref)
    assert case.status() == 0


def test_rope_toeplitz_rejects_bad_arguments():
    dev = torch.device("cuda")
    a = torch.zeros(3, dtype=torch.float32, device=dev)
    out = torch.zeros(15, dtype=torch.float32, device=dev)
    L = bd.lib()
    s = torch.cuda.current_stream().cuda_stream
    assert L.flash_gau_rope_toeplitz_bias(a.data_ptr(), a.data_ptr(), 3, 8, 10000.0,
                                          out.data_ptr(), s) == bd.EINVAL  # odd m
    assert L.flash_gau_rope_toeplitz_bias(a.data_ptr(), a.data_ptr(), 2, 8, 1.0,
                                          out.data_ptr(), s) == bd.EINVAL  # base <= 1
    assert L.flash_gau_rope_toeplitz_bias(None, a.data_ptr(), 2, 8, 10000.0,
                                          out.data_ptr(), s) == bd.EINVAL


# ---------------------------------------------------------------- GlobalOnly
# The local term times local_scale ("Transformer Quality in Linear Time",
# section 4.4, the ablation that keeps only the global, linear part, is
# local_scale = 0).  For bf16 io with local_scale = 0 the attention kernel
# forms no scores at all; other values scale P in its relu^2 warps.
@pytest.mark.parametrize("shape,causal,dtype,local_scale", [
    ((2, 1024, 256, 512, 128, 256), True, "bf16", 0.0),
    ((2, 1024, 256, 512, 128, 256), False, "bf16", 0.0),
    ((1, 512, 128, 768, 128, 128), True, "bf16", 0.0),
    ((1, 1024, 256, 512, 128, 256), True, "bf16", 0.5),
    ((1, 512, 128, 256, 128, 512), False, "bf16", -1.5),
    ((2, 200, 48, 72, 40, 40), True, "fp32", 0.0),
    ((1, 192, 64, 96, 32, 64), False, "fp32", 0.0),
    ((2, 200, 48, 72, 40, 40), True, "fp32", 0.25),
])
def test_forward_with_scaled_local_term(shape, causal, dtype, local_scale):
    B, T, d, e, s, C = shape
    case = Case(B, T, d, e, s, C, causal, dtype, seed=51 + C, local_scale=local_scale)
    O = case.run()
    ref, _ = case.reference()
    assert rel_err(O, ref) <= TOL[dtype], rel_err(O, ref)
    assert case.status() == 0


def test_global_only_does_not_depend_on_the_local_inputs():
    """local_scale = 0 (bf16, tensor-core path): changing the relative
    position bias, which enters only the local term, leaves the output
    bit-identical."""
    B, T, d, e, s, C = 1, 512, 128, 256, 128, 256
    case = Case(B, T, d, e, s, C, True, "bf16", seed=77, local_scale=0.0)
    O1 = case.run()
    case.weights.relpos.normal_()
    O2 = case.run()
    assert np.array_equal(O1, O2)
