"""Host-side checks of the C ABI: the library builds, loads and exports every
function include/flash_gau.h declares; layouts and argument validation work
without a GPU (invalid calls return before touching CUDA)."""

import ctypes
import os
import re

import pytest

from efficient_attention_transformer_gb300 import build as buildmod
from efficient_attention_transformer_gb300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    buildmod.build()
    return bd.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "flash_gau.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flash_gau_\w+)\s*\(", text)))


def test_header_declarations_are_exported(L):
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    assert sorted(bd.EXPORTED) == declared
    for name in declared:
        assert hasattr(L, name), name


def test_version_and_strerror(L):
    assert L.flash_gau_version() >= 100
    for code in (bd.OK, bd.EINVAL, bd.ENOTSUP, bd.EWORKSPACE, bd.ECUDA, bd.EDEVICE, bd.ETIMEOUT):
        assert bd.strerror(code)
    assert bd.strerror(12345) == "unknown status"


def test_layout_offsets_aligned_and_sized(L):
    B, T, C, d, e, s = 2, 8192, 256, 768, 1536, 128
    lay = bd.workspace_layout(B, T, C, d, e, s, True, bd.BF16)
    order = ["status", "U", "V", "heads", "state", "prefix", "gated", "bias", "xn", "rope"]
    offs = [lay[k] for k in order]
    assert offs == sorted(offs)
    assert all(o % 256 == 0 for o in offs)
    M, G = B * T, T // C
    assert lay["V"] - lay["U"] >= M * e * 2
    assert lay["heads"] - lay["V"] >= M * e * 2
    assert lay["state"] - lay["heads"] >= 4 * M * s * 2
    assert lay["prefix"] - lay["state"] >= B * G * s * e * 2
    assert lay["gated"] - lay["prefix"] >= B * G * s * e * 2
    assert lay["bias"] - lay["gated"] >= M * e * 2
    assert lay["xn"] - lay["bias"] >= (2 * C - 1) * 4
    assert lay["rope"] - lay["xn"] >= M * d * 2
    assert lay["total_bytes"] - lay["rope"] >= T * (s // 2) * 4
    nc = bd.workspace_layout(B, T, C, d, e, s, False, bd.BF16)
    # one prefix per chunk either way: the segmented forward needs it non-causal too
    assert nc["gated"] - nc["prefix"] == lay["gated"] - lay["prefix"]


@pytest.mark.parametrize("args,code", [
    ((1, 100, 64, 64, 128, 32, 1, bd.FP32), bd.EINVAL),     # T % C != 0
    ((0, 128, 64, 64, 128, 32, 1, bd.FP32), bd.EINVAL),     # B == 0
    ((1, 128, 64, 64, 128, 32, 1, 7), bd.EINVAL),           # unknown dtype
    ((1, 256, 128, 768, 1000, 128, 1, bd.BF16), bd.ENOTSUP),  # e % 256
    ((1, 256, 128, 192, 1536, 128, 1, bd.BF16), bd.ENOTSUP),  # d % 128
    ((1, 256, 128, 768, 1536, 64, 1, bd.BF16), bd.ENOTSUP),   # s != 128
    ((1, 192, 64, 768, 1536, 128, 1, bd.BF16), bd.ENOTSUP),   # C % 128
    ((1, 256, 64, 64, 128, 256, 1, bd.FP32), bd.ENOTSUP),     # s > 128 (fp32)
])
def test_layout_rejects(L, args, code):
    lay = bd.WorkspaceLayout()
    assert L.flash_gau_workspace_layout_query(*args, ctypes.byref(lay)) == code


def test_forward_rejects_before_any_launch(L):
    w = bd.Weights(1, 2, 3, 4, 5, 64, 128, 32, 1.0, 1.0)  # fake non-null pointers
    ws = 1 << 20
    # null X
    assert L.flash_gau_forward(None, ctypes.byref(w), 1, 256, 64, 1, bd.FP32, 8, 256 * 64,
                               ws, None) == bd.EINVAL
    # null weights
    assert L.flash_gau_forward(16, None, 1, 256, 64, 1, bd.FP32, 8, 256, ws, None) == bd.EINVAL
    # ragged T
    assert L.flash_gau_forward(16, ctypes.byref(w), 1, 250, 64, 1, bd.FP32, 1 << 40, 256,
                               ws, None) == bd.EINVAL
    # workspace too small
    assert L.flash_gau_forward(16, ctypes.byref(w), 1, 256, 64, 1, bd.FP32, 1 << 40, 256,
                               16, None) == bd.EWORKSPACE
    # misaligned workspace
    assert L.flash_gau_forward(16, ctypes.byref(w), 1, 256, 64, 1, bd.FP32, 1 << 40, 257,
                               ws, None) == bd.EWORKSPACE
    # output overlapping X
    assert L.flash_gau_forward(1 << 30, ctypes.byref(w), 1, 256, 64, 1, bd.FP32,
                               (1 << 30) + 64, 1 << 34, ws, None) == bd.EINVAL
    # events requested but none given
    assert L.flash_gau_forward_timed(16, ctypes.byref(w), 1, 256, 64, 1, bd.FP32, 1 << 40,
                                     256, ws, None, None, 3) == bd.EINVAL


def test_workspace_bytes_matches_layout(L):
    w = bd.Weights(1, 2, 3, 4, 5, 768, 1536, 128, 1.0, 1.0)
    n = L.flash_gau_workspace_bytes(8, 1024, 256, ctypes.byref(w), 1, bd.BF16)
    assert n == bd.workspace_layout(8, 1024, 256, 768, 1536, 128, True, bd.BF16)["total_bytes"]
    assert L.flash_gau_workspace_bytes(8, 1000, 256, ctypes.byref(w), 1, bd.BF16) == 0


def test_stage_names(L):
    for dt in (bd.FP32, bd.BF16):
        names = bd.stage_names(dt, True)
        assert len(names) == bd.num_stages(dt, True) >= 1
        assert L.flash_gau_stage_name(dt, 1, len(names)) is None


@pytest.mark.parametrize("opts", [
    dict(norm=7),                                   # unknown norm
    dict(norm=bd.NORM_LAYER, norm_g=None),          # missing scale
    dict(norm=bd.NORM_LAYER, norm_eps=0.0),         # eps <= 0
    dict(rope=1, rope_base=1.0),                    # base <= 1
    dict(pos_offset=-1),                            # negative position
])
def test_block_forward_rejects_bad_options_before_any_launch(L, opts):
    w = bd.Weights(1, 2, 3, 4, 5, 128, 256, 128, 1.0, 1.0)
    base = dict(norm=bd.NORM_LAYER, norm_g=6, norm_b=None, norm_eps=1e-5, rope=1,
                rope_base=10000.0, pos_offset=0, residual=1)
    base.update(opts)
    blk = bd.Block(base["norm"], base["norm_g"], base["norm_b"], base["norm_eps"], base["rope"],
                   base["rope_base"], base["pos_offset"], base["residual"])
    n = bd.workspace_layout(1, 256, 128, 128, 256, 128, True, bd.BF16)["total_bytes"]
    assert L.flash_gau_block_forward(16, ctypes.byref(w), ctypes.byref(blk), 1, 256, 128, 1,
                                     bd.BF16, 1 << 40, 256, n, None) == bd.EINVAL
    assert L.flash_gau_block_forward(16, ctypes.byref(w), None, 1, 256, 128, 1, bd.BF16,
                                     1 << 40, 256, n, None) == bd.EINVAL


def test_block_forward_rejects_rope_with_odd_head_width(L):
    w = bd.Weights(1, 2, 3, 4, 5, 64, 128, 33, 1.0, 1.0)
    blk = bd.Block(bd.NORM_NONE, None, None, 1e-5, 1, 10000.0, 0, 1)
    n = bd.workspace_layout(1, 256, 64, 64, 128, 33, True, bd.FP32)["total_bytes"]
    assert L.flash_gau_block_forward(16, ctypes.byref(w), ctypes.byref(blk), 1, 256, 64, 1,
                                     bd.FP32, 1 << 40, 256, n, None) == bd.EINVAL


@pytest.mark.parametrize("lin,loc", [(float("inf"), 1.0), (1.0, float("nan")),
                                     (1.0, float("-inf"))])
def test_non_finite_term_factors_rejected_before_any_launch(L, lin, loc):
    """An infinite or NaN factor on either term is refused on the host by the
    forward, the backward and the decode step."""
    w = bd.Weights(1, 2, 3, 4, 5, 64, 128, 32, lin, loc)
    ws = 1 << 20
    assert L.flash_gau_forward(16, ctypes.byref(w), 1, 256, 64, 1, bd.FP32, 1 << 40, 256,
                               ws, None) == bd.EINVAL
    g = bd.Grads(1, 2, 3, 4, 5, 6)
    assert L.flash_gau_backward(16, 32, ctypes.byref(w), 1, 256, 64, 1, bd.FP32,
                                ctypes.byref(g), 256, ws, None) == bd.EINVAL
    assert L.flash_gau_decode_step(16, ctypes.byref(w), 1, 64, bd.FP32, 256, ws, 1 << 40,
                                   None) == bd.EINVAL


def test_product_and_oracle_share_no_code():
    """The CUDA path never imports the oracle, and the oracle never imports
    the package: the two sides share only the seeded input generator."""
    pkg = os.path.join(ROOT, "efficient_attention_transformer_gb300")
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f), errors="replace").read()
                assert not pat.search(text), f
                assert "oracle/" not in text, f
    opat = re.compile(r"efficient_attention_transformer_gb300\.(?!synthetic)")
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith(".py"):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert not opat.search(text), f


def test_missing_library_fails_loudly(monkeypatch):
    """Without the built library every entry point raises; nothing falls
    back to a CPU computation."""
    import torch
    monkeypatch.setattr(bd, "_LIB_PATH", os.path.join(ROOT, "no_such_dir", "libflashgau.so"))
    monkeypatch.setattr(bd, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        bd.lib()
    # host tensors are refused as weights: there is no CPU path to take them
    with pytest.raises(ValueError, match="CUDA tensor"):
        bd.GauWeights(torch.zeros(64, 288), torch.zeros(128, 64), torch.zeros(4, 32),
                      torch.zeros(4, 32), torch.zeros(127), 64, 128, 32)


def test_host_forward_and_segmented_forward_reject_before_any_launch(L):
    w = bd.Weights(1, 2, 3, 4, 5, 64, 128, 32, 1.0, 1.0)
    n = L.flash_gau_forward_host_workspace_bytes(2, 256, 64, ctypes.byref(w), 1, bd.FP32)
    assert n > 0
    # ragged T: no workspace size, and the call refuses
    assert L.flash_gau_forward_host_workspace_bytes(2, 250, 64, ctypes.byref(w), 1, bd.FP32) == 0
    assert L.flash_gau_forward_host(16, ctypes.byref(w), 2, 250, 64, 1, bd.FP32, 32, 256, n,
                                    None) == bd.EINVAL
    # null host buffers, too small or misaligned workspace
    assert L.flash_gau_forward_host(None, ctypes.byref(w), 2, 256, 64, 1, bd.FP32, 32, 256, n,
                                    None) == bd.EINVAL
    assert L.flash_gau_forward_host(16, ctypes.byref(w), 2, 256, 64, 1, bd.FP32, 32, 256, n - 1,
                                    None) == bd.EWORKSPACE
    assert L.flash_gau_forward_host(16, ctypes.byref(w), 2, 256, 64, 1, bd.FP32, 32, 257, n,
                                    None) == bd.EWORKSPACE
    # the segmented forward validates like the plain one
    seg = bd.Segments(None, 1)
    assert L.flash_gau_forward_segmented(None, ctypes.byref(w), ctypes.byref(seg), 1, 256, 64, 1,
                                         bd.FP32, 1 << 40, 256, 1 << 20, None) == bd.EINVAL
    assert L.flash_gau_forward_segmented(16, ctypes.byref(w), ctypes.byref(seg), 1, 250, 64, 1,
                                         bd.FP32, 1 << 40, 256, 1 << 20, None) == bd.EINVAL
