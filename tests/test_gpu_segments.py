"""GPU parity of the chunk-masked global term (flash_gau_forward_segmented):
segment ids for packed text and the row-normalised mask ("Transformer
Quality in Linear Time", Paper vs code and Pitfalls, the segment-mask
items), against the float64 oracle's ``chunk_mask`` reading on the same
seeded inputs, with the layer's tolerances (1e-4 of the maximum for fp32
io, 2e-2 for bf16 io; the prefix states, stored in the io type, 1e-2)."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from gpu_harness import Case, TOL, TOL_INTER, rel_err, unblock64
from oracle import flash_gau

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


def _ids(kind, B, G, seed):
    rng = np.random.default_rng(seed)
    if kind is None:
        return None
    if kind == "runs":  # packed documents: non-decreasing ids, random run lengths
        out = np.zeros((B, G), dtype=np.int32)
        for b in range(B):
            cuts = np.sort(rng.choice(np.arange(1, G), size=min(2, G - 1), replace=False))
            for c in cuts:
                out[b, c:] += 1
        return out
    if kind == "distinct":
        return np.tile(np.arange(G, dtype=np.int32), (B, 1))
    if kind == "gap":  # an id that comes back after another: a new segment
        out = np.zeros((B, G), dtype=np.int32)
        out[:, G // 3:2 * G // 3] = 9
        return out
    raise ValueError(kind)


def _check(shape, causal, dtype, kind, average, seed):
    B, T, d, e, s, C = shape
    G = T // C
    case = Case(B, T, d, e, s, C, causal, dtype, seed=seed)
    ids = _ids(kind, B, G, seed + 1)
    tids = None if ids is None else torch.tensor(ids, dtype=torch.int32, device="cuda")
    bd.forward_segmented(case.X, case.weights, C, causal, tids, average, out=case.out,
                         workspace=case.workspace)
    torch.cuda.synchronize()
    O = case.out.double().cpu().numpy()
    i = case.inp
    ref, inter = flash_gau(i["X"], i["W_u"], i["W_v"], i["W_z"], i["W_o"], i["gamma"],
                           i["beta"], i["relpos"], C, causal, segment_ids=ids,
                           chunk_average=average)
    err = rel_err(O, ref)
    # the prefix states as the attention reads them: one per chunk when
    # causal or segmented, else one per batch row
    per_chunk = causal or ids is not None
    rows = (B * G if per_chunk else B) * s
    tdt = case.X.dtype
    raw = case.workspace[case.layout["prefix"]:]
    n = rows * e
    pre = raw[: n * (2 if tdt == torch.bfloat16 else 4)].view(tdt).double().cpu().numpy()
    if tdt == torch.bfloat16:
        pre = unblock64(pre, rows, e)
    pre = pre.reshape(-1, s, e)
    want = inter["prefix"].reshape(B * G, s, e) if per_chunk else inter["prefix"][:, 0]
    pre_err = rel_err(pre, want)
    print(dtype, causal, kind, average, "O %.2e prefix %.2e" % (err, pre_err))
    assert err <= TOL[dtype], err
    assert pre_err <= TOL_INTER[dtype], pre_err
    assert case.status() == 0


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kind,average", [("runs", False), ("runs", True), ("gap", True),
                                          ("distinct", False), (None, True)])
def test_segmented_bf16_tensor_core_path(causal, kind, average):
    _check((2, 2048, 256, 512, 128, 256), causal, "bf16", kind, average, seed=101)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kind,average", [("runs", False), ("runs", True), ("gap", False),
                                          ("distinct", True), (None, True)])
def test_segmented_fp32_path(causal, kind, average):
    _check((2, 240, 48, 72, 40, 24), causal, "fp32", kind, average, seed=111)


def test_segmented_without_mask_equals_the_plain_forward():
    """seg = NULL through the segmented entry point is flash_gau_forward,
    bit for bit."""
    case = Case(1, 1024, 256, 512, 128, 256, False, "bf16", seed=121)
    O1 = case.run()
    bd.forward_segmented(case.X, case.weights, 256, False, None, False, out=case.out,
                         workspace=case.workspace)
    torch.cuda.synchronize()
    assert np.array_equal(O1, case.out.double().cpu().numpy())


def test_segment_ids_shape_is_checked():
    case = Case(1, 512, 256, 512, 128, 256, True, "bf16", seed=122)
    bad = torch.zeros(1, 3, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        bd.forward_segmented(case.X, case.weights, 256, True, bad)
