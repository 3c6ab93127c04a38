"""Pins for the float64 oracle, each against something other than the oracle
itself: library routines, hand-derived golden fixtures, a scalar per-token
formulation, the pages' associativity and cumulative-sum arguments, special
cases that reduce the layer to a GLU or to FLASH-Quad, and invariants.
CPU only."""

import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

from oracle import flash_gau, relpos_bias, swish, algorithmic_flops_per_token
from efficient_attention_transformer_gb300.synthetic import (
    make_inputs, round_bf16)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_index_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(t) for t in line.split()])
    return np.array(rows)


def _run(inp, C, causal, lin_scale=1.0):
    return flash_gau(inp["X"], inp["W_u"], inp["W_v"], inp["W_z"], inp["W_o"],
                     inp["gamma"], inp["beta"], inp["relpos"], C, causal,
                     lin_scale)


# ---------------------------------------------------------------- swish ----

def test_swish_matches_scipy_expit():
    x = np.concatenate([np.linspace(-30, 30, 2001), [0.0, -745.0, 800.0]])
    ref = x * scipy.special.expit(x)
    np.testing.assert_allclose(swish(x), ref, rtol=1e-14, atol=1e-300)
    assert swish(0.0) == 0.0


# ---------------------------------------------------- relative position ----

@pytest.mark.parametrize("n,name", [(3, "relpos_toeplitz_n3.txt"),
                                    (5, "relpos_toeplitz_n5.txt")])
def test_relpos_golden_from_code4(n, name):
    idx = _load_index_table(name)
    w = np.arange(2 * n - 1, dtype=np.float64)
    np.testing.assert_array_equal(relpos_bias(w, n), idx.astype(np.float64))


@pytest.mark.parametrize("n", [1, 2, 7, 64])
def test_relpos_matches_scipy_toeplitz(n):
    w = np.random.default_rng(n).standard_normal(2 * n - 1)
    # first column b[i, 0] = w[n-1-i]; first row b[0, j] = w[n-1+j]
    ref = scipy.linalg.toeplitz(w[n - 1::-1], w[n - 1:])
    np.testing.assert_array_equal(relpos_bias(w, n), ref)


# ------------------------------------------------- scalar token loop -------

def _brute_force(inp, C, causal, lin_scale):
    """Per-token scalar restatement: every output element summed from its
    inputs with Python floats; the global term is token-level linear
    attention over tokens of strictly earlier chunks (causal) or all chunks
    (non-causal), never through chunk states."""
    X, Wu, Wv, Wz, Wo = (inp[k].tolist() for k in ("X", "W_u", "W_v", "W_z", "W_o"))
    ga, be, rp = inp["gamma"].tolist(), inp["beta"].tolist(), inp["relpos"].tolist()
    B, T, d = inp["X"].shape
    e, s = inp["W_u"].shape[1], inp["W_z"].shape[1]

    def sw(a):
        return a / (1.0 + math.exp(-a))

    def proj(x, W, n):
        return [sw(sum(x[k] * W[k][j] for k in range(d))) for j in range(n)]

    O = np.zeros((B, T, d))
    for b in range(B):
        u = [proj(X[b][t], Wu, e) for t in range(T)]
        v = [proj(X[b][t], Wv, e) for t in range(T)]
        z = [proj(X[b][t], Wz, s) for t in range(T)]
        head = [[[z[t][k] * ga[h][k] + be[h][k] for k in range(s)]
                 for t in range(T)] for h in range(4)]
        qq, kq, ql, kl = head
        for t in range(T):
            g, i = divmod(t, C)
            mix = [0.0] * e
            for j in range(C):
                if causal and j > i:
                    continue
                tj = g * C + j
                sc = sum(qq[t][k] * kq[tj][k] for k in range(s)) / C + rp[j - i + C - 1]
                a = max(sc, 0.0) ** 2
                for c in range(e):
                    mix[c] += a * v[tj][c]
            for tp in range(T):
                gp = tp // C
                if causal and gp >= g:
                    continue
                w = lin_scale * sum(ql[t][k] * kl[tp][k] for k in range(s))
                for c in range(e):
                    mix[c] += w * v[tp][c]
            for o in range(d):
                O[b, t, o] = sum(u[t][c] * mix[c] * Wo[c][o] for c in range(e))
    return O


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("T,C", [(12, 4), (6, 6), (8, 2)])
def test_oracle_matches_scalar_token_loop(causal, T, C):
    inp = make_inputs(B=2, T=T, d=3, e=5, s=2, C=C, dtype="fp32", seed=7)
    # larger head scales so relu^2 is active on some pairs and off on others
    inp["gamma"] = inp["gamma"] * 3.0
    O, _ = _run(inp, C, causal, lin_scale=0.5)
    ref = _brute_force(inp, C, causal, lin_scale=0.5)
    np.testing.assert_allclose(O, ref, rtol=1e-11, atol=1e-12)


# --------------------------------------------- special cases of the layer --

def test_attention_identity_reduces_to_glu():
    """A = I turns GAU into a GLU with Swish on both branches ("Gated
    Attention" / "Joining Forces": O = (U * V) W_o).  A = I is reached through
    the parameters: zero quadratic heads make Q K^T = 0, and a bias that is 1
    on the diagonal and -1 elsewhere gives relu^2(b) = I; a zero linear query
    removes the global term."""
    C = 8
    inp = make_inputs(B=2, T=32, d=16, e=24, s=8, C=C, dtype="fp32", seed=3)
    inp["gamma"][[0, 1, 2]] = 0.0
    inp["beta"][[0, 1, 2]] = 0.0
    inp["relpos"] = -np.ones(2 * C - 1)
    inp["relpos"][C - 1] = 1.0
    for causal in (True, False):
        O, _ = _run(inp, C, causal)
        X = inp["X"]
        hu, hv = X @ inp["W_u"], X @ inp["W_v"]
        glu = (hu * scipy.special.expit(hu)) * (hv * scipy.special.expit(hv))
        np.testing.assert_allclose(O, glu @ inp["W_o"], rtol=1e-12, atol=1e-13)


def test_causal_first_chunk_has_no_global_term():
    C = 16
    inp = make_inputs(B=3, T=64, d=8, e=12, s=4, C=C, dtype="fp32", seed=5)
    _, it = _run(inp, C, True)
    assert np.all(it["prefix"][:, 0] == 0.0)
    assert np.all(it["Vl"][:, :C] == 0.0)
    assert np.any(it["Vl"][:, C:] != 0.0)


def test_noncausal_global_term_is_full_linear_attention():
    """Eq. 7 summed over chunks equals linear attention applied to the whole
    sequence, (Q_lin K_lin^T) V ("Mixed Chunking": exactly equivalent)."""
    C = 8
    inp = make_inputs(B=2, T=40, d=8, e=12, s=6, C=C, dtype="fp32", seed=11)
    _, it = _run(inp, C, False, lin_scale=0.25)
    Ql, Kl = it["heads"][2], it["heads"][3]
    for b in range(2):
        ref = 0.25 * (Ql[b] @ Kl[b].T) @ it["V"][b]
        np.testing.assert_allclose(it["Vl"][b], ref, rtol=1e-11, atol=1e-11)


def test_causal_global_term_is_token_cumsum_at_chunk_ends():
    """Eq. 8 equals token-level linear attention read at the end of the
    previous chunk: M_t = M_{t-1} + K_t V_t^T (the cumulative-sum form of
    section 3.1), and chunk g reads M at token gC - 1."""
    C = 4
    inp = make_inputs(B=2, T=24, d=6, e=7, s=5, C=C, dtype="fp32", seed=13)
    _, it = _run(inp, C, True)
    Ql, Kl, V = it["heads"][2], it["heads"][3], it["V"]
    for b in range(2):
        M = np.cumsum(Kl[b][:, :, None] * V[b][:, None, :], axis=0)  # [T, s, e]
        for t in range(24):
            g = t // C
            ref = np.zeros(7) if g == 0 else Ql[b, t] @ M[g * C - 1]
            np.testing.assert_allclose(it["Vl"][b, t], ref, rtol=1e-11, atol=1e-11)


def test_noncausal_invariant_to_chunk_permutation():
    """Local attention stays inside a chunk and eq. 7's global sum is
    order-free, so permuting whole chunks of the input permutes the output
    the same way."""
    C, G = 8, 5
    inp = make_inputs(B=2, T=C * G, d=8, e=10, s=4, C=C, dtype="fp32", seed=17)
    O, _ = _run(inp, C, False)
    perm = np.array([3, 0, 4, 2, 1])
    rows = np.concatenate([np.arange(p * C, (p + 1) * C) for p in perm])
    inp2 = dict(inp, X=inp["X"][:, rows])
    O2, _ = _run(inp2, C, False)
    np.testing.assert_allclose(O2, O[:, rows], rtol=1e-11, atol=1e-12)
    # causal is NOT invariant: the global term depends on chunk order
    Oc, _ = _run(inp, C, True)
    Oc2, _ = _run(inp2, C, True)
    assert not np.allclose(Oc2, Oc[:, rows])


def test_zero_quadratic_heads_leave_only_global_term():
    C = 8
    inp = make_inputs(B=1, T=32, d=8, e=10, s=4, C=C, dtype="fp32", seed=19)
    inp["gamma"][[0, 1]] = 0.0
    inp["beta"][[0, 1]] = 0.0
    inp["relpos"][:] = 0.0
    O, it = _run(inp, C, True)
    assert np.all(it["Vq"] == 0.0)
    np.testing.assert_allclose(O, (it["U"] * it["Vl"]) @ inp["W_o"], rtol=1e-13)


def test_large_negative_bias_switches_relu2_off():
    C = 8
    inp = make_inputs(B=1, T=16, d=8, e=6, s=4, C=C, dtype="fp32", seed=23)
    inp["relpos"][:] = -1e3
    _, it = _run(inp, C, False)
    assert np.all(it["Vq"] == 0.0)


def test_local_only_and_lin_scale_linearity():
    C = 8
    inp = make_inputs(B=2, T=32, d=8, e=10, s=4, C=C, dtype="fp32", seed=29)
    O0, it0 = _run(inp, C, True, lin_scale=0.0)
    assert np.all(it0["Vl"] == 0.0)
    np.testing.assert_allclose(O0, (it0["U"] * it0["Vq"]) @ inp["W_o"], rtol=1e-13)
    _, it1 = _run(inp, C, True, lin_scale=1.0)
    _, it3 = _run(inp, C, True, lin_scale=3.0)
    np.testing.assert_allclose(it3["Vl"], 3.0 * it1["Vl"], rtol=1e-12)


def test_relu2_weights_nonnegative_and_masked():
    C = 16
    inp = make_inputs(B=1, T=32, d=8, e=6, s=4, C=C, dtype="fp32", seed=31)
    inp["gamma"] = inp["gamma"] * 4.0
    from oracle import chunk_scores, relpos_bias as rb
    _, it = _run(inp, C, True)
    a = chunk_scores(it["heads"][0][0, :C], it["heads"][1][0, :C],
                     rb(inp["relpos"], C), C, True)
    assert np.all(a >= 0.0)
    assert np.all(np.triu(a, 1) == 0.0)
    assert np.any(np.diag(a) > 0.0)


def test_chunk_of_whole_sequence_causal_has_no_global_term():
    """C = T: the layer degenerates to FLASH-Quad (appendix C.3), whose causal
    output has no linear term at all."""
    T = 16
    inp = make_inputs(B=2, T=T, d=8, e=6, s=4, C=T, dtype="fp32", seed=37)
    O, it = _run(inp, T, True)
    assert np.all(it["Vl"] == 0.0)
    np.testing.assert_allclose(O, (it["U"] * it["Vq"]) @ inp["W_o"], rtol=1e-13)


def test_rejects_ragged_length():
    inp = make_inputs(B=1, T=10, d=4, e=4, s=2, C=4, dtype="fp32", seed=0)
    with pytest.raises(ValueError):
        _run(inp, 4, True)


# ------------------------------------------------------------ FLOP count --

def test_flop_count_matches_operation_count():
    """Counts multiply-adds of the tiny scalar formulation directly."""
    d, e, s, C = 3, 5, 2, 4
    for causal in (True, False):
        visible = sum((i + 1) if causal else C for i in range(C)) / C
        per_token = 2 * (d * (2 * e + s) + e * d + visible * s + visible * e + 2 * s * e)
        assert algorithmic_flops_per_token(d, e, s, C, causal) == pytest.approx(per_token)
    assert algorithmic_flops_per_token(768, 1536, 128, 256, True) == 8488576.0


def test_bf16_rounding_is_nearest_even():
    import torch
    x = np.random.default_rng(0).standard_normal(10000) * 100
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(round_bf16(x), ref)


# ------------------------------------------------- flash_block: norm, RoPE --

from oracle import flash_block, layer_norm, rope, scale_norm  # noqa: E402


def test_rope_golden_worked_example():
    """Hand-worked rotation of one 4-wide vector (tests/golden)."""
    want = None
    with open(os.path.join(GOLDEN, "rope_s4_base10000.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                want = np.array([float(t) for t in line.split()])
    got = rope(np.array([[1.0, 2.0, 3.0, 4.0]]), np.array([100.0]), 10000.0)[0]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_rope_equals_complex_rotation_and_keeps_norms():
    """Pairs as complex numbers h2i + i h2i+1 multiplied by e^(i p theta_i),
    theta_i = base^(-2i/s): an independent formulation.  Rotations keep each
    pair's length, and position 0 is the identity."""
    rng = np.random.default_rng(3)
    T, s, base = 9, 8, 500.0
    h = rng.normal(size=(2, T, s))
    pos = rng.uniform(0, 50, size=T)
    z = h[..., 0::2] + 1j * h[..., 1::2]
    theta = base ** (-2.0 * np.arange(s // 2) / s)
    zr = z * np.exp(1j * pos[:, None] * theta[None, :])
    ref = np.empty_like(h)
    ref[..., 0::2], ref[..., 1::2] = zr.real, zr.imag
    got = rope(h, pos, base)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.abs(got[..., 0::2] + 1j * got[..., 1::2]), np.abs(z),
                               rtol=1e-12)
    np.testing.assert_allclose(rope(h, np.zeros(T), base), h, rtol=0, atol=0)


def test_rope_scores_depend_on_relative_position_only():
    """<rope(q, m), rope(k, n)> = <rope(q, m + d), rope(k, n + d)>."""
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=(1, 6)), rng.normal(size=(1, 6))
    for m, n, dlt in [(3, 7, 11), (0, 5, 100), (40, 2, -30)]:
        a = rope(q, np.array([m]))[0] @ rope(k, np.array([n]))[0]
        b = rope(q, np.array([m + dlt]))[0] @ rope(k, np.array([n + dlt]))[0]
        assert abs(a - b) < 1e-12


def test_layer_norm_matches_torch_and_scale_norm_sets_the_length():
    import torch
    rng = np.random.default_rng(5)
    x = rng.normal(1.5, 3.0, size=(4, 7, 24))
    g, b = rng.normal(1, 0.1, 24), rng.normal(0, 0.1, 24)
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (24,), torch.tensor(g),
                                         torch.tensor(b), eps=1e-5).numpy()
    np.testing.assert_allclose(layer_norm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)
    y = scale_norm(x, 2.5)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 2.5, rtol=1e-12)


def _brute_force_block(inp, C, causal, lin_scale, pos_offset, base):
    """Scalar restatement of the block with RoPE and no norm: the heads of
    each token are rotated as complex numbers at the token's global position,
    the global term is token-level linear attention (never chunk states), and
    the residual is added per element."""
    X = inp["X"]
    B, T, d = X.shape
    e, s = inp["W_u"].shape[1], inp["W_z"].shape[1]
    Xl, Wu, Wv, Wz, Wo = (inp[k].tolist() for k in ("X", "W_u", "W_v", "W_z", "W_o"))
    ga, be, rp = inp["gamma"].tolist(), inp["beta"].tolist(), inp["relpos"].tolist()

    def sw(a):
        return a / (1.0 + math.exp(-a))

    def proj(x, W, n):
        return [sw(sum(x[k] * W[k][j] for k in range(d))) for j in range(n)]

    def rot(vec, p):
        out = []
        for i in range(s // 2):
            z = complex(vec[2 * i], vec[2 * i + 1]) * complex(
                math.cos(p * base ** (-2.0 * i / s)), math.sin(p * base ** (-2.0 * i / s)))
            out += [z.real, z.imag]
        return out

    Y = np.zeros((B, T, d))
    for b in range(B):
        u = [proj(Xl[b][t], Wu, e) for t in range(T)]
        v = [proj(Xl[b][t], Wv, e) for t in range(T)]
        z = [proj(Xl[b][t], Wz, s) for t in range(T)]
        head = [[rot([z[t][k] * ga[h][k] + be[h][k] for k in range(s)], t + pos_offset)
                 for t in range(T)] for h in range(4)]
        qq, kq, ql, kl = head
        for t in range(T):
            g, i = divmod(t, C)
            mix = [0.0] * e
            for j in range(C):
                if causal and j > i:
                    continue
                tj = g * C + j
                sc = sum(qq[t][k] * kq[tj][k] for k in range(s)) / C + rp[j - i + C - 1]
                a = max(sc, 0.0) ** 2
                for c in range(e):
                    mix[c] += a * v[tj][c]
            for tp in range(T):
                if causal and tp // C >= g:
                    continue
                w = lin_scale * sum(ql[t][k] * kl[tp][k] for k in range(s))
                for c in range(e):
                    mix[c] += w * v[tp][c]
            for o in range(d):
                Y[b, t, o] = Xl[b][t][o] + sum(u[t][c] * mix[c] * Wo[c][o] for c in range(e))
    return Y


def _block(inp, C, causal, **kw):
    return flash_block(inp["X"], inp["W_u"], inp["W_v"], inp["W_z"], inp["W_o"],
                       inp["gamma"], inp["beta"], inp["relpos"], C, causal, **kw)[0]


@pytest.mark.parametrize("causal", [True, False])
def test_block_matches_scalar_loop_with_global_rope_positions(causal):
    """RoPE at global positions (not restarted per chunk) reaches the global
    term through Q_lin K_lin^T across chunks; the token loop pins that."""
    inp = make_inputs(B=1, T=8, d=3, e=4, s=4, C=4, dtype="fp32", seed=8)
    inp["gamma"] = inp["gamma"] * 3.0
    Y = _block(inp, 4, causal, lin_scale=0.5, norm=None, rope_base=7.0, pos_offset=3)
    ref = _brute_force_block(inp, 4, causal, 0.5, 3, 7.0)
    np.testing.assert_allclose(Y, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_block_invariant_to_global_position_shift(causal):
    """Positions enter only through rotations of both sides of every score, so
    shifting all of them changes nothing."""
    inp = make_inputs(B=2, T=16, d=8, e=12, s=8, C=4, dtype="fp32", seed=9)
    g, b = np.ones(8), np.zeros(8)
    a = _block(inp, 4, causal, norm="layer", norm_g=g, norm_b=b, pos_offset=0)
    c = _block(inp, 4, causal, norm="layer", norm_g=g, norm_b=b, pos_offset=1234)
    np.testing.assert_allclose(a, c, rtol=1e-10, atol=1e-10)


def test_block_is_residual_around_the_layer_of_the_normalised_input():
    """Without RoPE: Y - X = flash_gau(LayerNorm(X)), LayerNorm taken from
    torch; with RoPE off and no norm it is X + flash_gau(X)."""
    import torch
    inp = make_inputs(B=2, T=8, d=6, e=8, s=4, C=4, dtype="fp32", seed=10)
    rng = np.random.default_rng(11)
    g, b = rng.normal(1, 0.1, 6), rng.normal(0, 0.1, 6)
    Xn = torch.nn.functional.layer_norm(torch.tensor(inp["X"], dtype=torch.float64), (6,),
                                        torch.tensor(g), torch.tensor(b), eps=1e-5).numpy()
    Y = _block(inp, 4, True, norm="layer", norm_g=g, norm_b=b, rope_on=False)
    ref, _ = flash_gau(Xn, inp["W_u"], inp["W_v"], inp["W_z"], inp["W_o"], inp["gamma"],
                       inp["beta"], inp["relpos"], 4, True)
    np.testing.assert_allclose(Y - inp["X"], ref, rtol=1e-10, atol=1e-12)
    Y0 = _block(inp, 4, True, norm=None, rope_on=False)
    np.testing.assert_allclose(Y0 - inp["X"], _run(inp, 4, True)[0], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- RoPE-Toeplitz bias
import oracle as O  # noqa: E402
import oracle as O_  # noqa: E402
def test_rope_toeplitz_golden_worked_example():
    """Hand-worked 3 x 3 bias from a = (1, 0), b = (0, 1) (tests/golden)."""
    with open(os.path.join(GOLDEN, "rope_toeplitz_m2_n3.txt")) as f:
        want = np.array([[float(x) for x in ln.split()] for ln in f
                         if ln.strip() and not ln.startswith("#")])
    got = O.rope_toeplitz_bias(np.array([1.0, 0.0]), np.array([0.0, 1.0]), 3)
    assert np.allclose(got, want, rtol=0, atol=1e-15)


def test_rope_toeplitz_depends_on_offset_only():
    """Rotations compose (R(i)^T R(j) = R(j - i)), so the bias is Toeplitz:
    every diagonal is constant, for any vectors and base."""
    rng = np.random.default_rng(21)
    for m, n, base in [(8, 9, 10000.0), (128, 40, 10000.0), (6, 17, 37.0)]:
        T = O.rope_toeplitz_bias(rng.normal(size=m), rng.normal(size=m), n, base)
        assert np.allclose(T[1:, 1:], T[:-1, :-1], rtol=0, atol=1e-12)
        # and it is not symmetric in general (a and b play different roles)
        assert not np.allclose(T, T.T)


def test_rope_toeplitz_diagonal_is_inner_product():
    """On the diagonal both copies turn by the same angle: bias[i, i] = a . b."""
    rng = np.random.default_rng(22)
    a, b = rng.normal(size=128), rng.normal(size=128)
    T = O.rope_toeplitz_bias(a, b, 33)
    assert np.allclose(np.diag(T), a @ b, rtol=1e-12, atol=1e-12)


def test_toeplitz_relpos_round_trip():
    """Reading the table back and rebuilding the matrix with relpos_bias
    gives the same matrix (the layer's bias index rule, pinned by the Code 4
    fixtures, is the inverse)."""
    rng = np.random.default_rng(23)
    T = O.rope_toeplitz_bias(rng.normal(size=16), rng.normal(size=16), 12)
    rp = O.toeplitz_relpos(T)
    assert rp.shape == (23,)
    assert np.allclose(O.relpos_bias(rp, 12), T, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- backward
@pytest.mark.parametrize("causal,lin_scale,C,local_scale", [
    (True, 1.0, 4, 1.0), (False, 1.0, 4, 1.0), (True, 0.25, 2, 0.5), (False, 0.0, 8, 1.0),
    (True, 1.0, 4, 0.0)])
def test_backward_matches_finite_differences(causal, lin_scale, C, local_scale):
    """Every gradient entry of L = sum(dO * O) against central differences of
    the forward oracle (step 1e-6, float64), on a problem small enough to
    perturb each input and parameter once."""
    rng = np.random.default_rng(51 + C)
    B, T, d, e, s = 2, 8, 4, 6, 4
    args = dict(
        X=rng.normal(size=(B, T, d)), W_u=rng.normal(size=(d, e)) / 2,
        W_v=rng.normal(size=(d, e)) / 2, W_z=rng.normal(size=(d, s)) / 2,
        W_o=rng.normal(size=(e, d)) / 2, gamma=rng.normal(1.0, 0.3, (4, s)),
        beta=rng.normal(0.0, 0.3, (4, s)), relpos=rng.normal(0.0, 0.5, 2 * C - 1))
    dO = rng.normal(size=(B, T, d))

    def loss(a):
        O, _ = flash_gau(a["X"], a["W_u"], a["W_v"], a["W_z"], a["W_o"], a["gamma"],
                         a["beta"], a["relpos"], C, causal, lin_scale, local_scale=local_scale)
        return float(np.sum(dO * O))

    grads = O.flash_gau_backward(args["X"], args["W_u"], args["W_v"], args["W_z"], args["W_o"],
                                 args["gamma"], args["beta"], args["relpos"], C, causal, dO,
                                 lin_scale, local_scale)
    h = 1e-6
    for name in args:
        g = grads["d" + name]
        assert g.shape == args[name].shape
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            plus = {k: v.copy() for k, v in args.items()}
            minus = {k: v.copy() for k, v in args.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            num[idx] = (loss(plus) - loss(minus)) / (2 * h)
        scale = max(1.0, float(np.max(np.abs(num))))
        assert np.max(np.abs(num - g)) <= 1e-6 * scale, (name, np.max(np.abs(num - g)))


def test_swish_grad_against_library_derivative():
    """swish'(x) = d/dx [x * expit(x)] computed with scipy's expit and the
    product rule on a grid, including large |x|."""
    x = np.linspace(-30, 30, 1201)
    sg = scipy.special.expit(x)
    want = sg + x * sg * (1 - sg)
    assert np.allclose(O.swish_grad(x), want, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("C,T,lin_scale,local_scale", [
    (4, 11, 1.0, 1.0), (8, 24, 0.5, 1.0), (1, 5, 1.0, 1.0), (16, 7, 0.0, 1.0), (4, 13, 1.0, 0.0)])
def test_decode_steps_equal_causal_forward_rows(C, T, lin_scale, local_scale):
    """By causality, the decode step's output for token t is row t of the
    causal forward over any sequence that starts with the same t + 1
    tokens (the rest zero-padded to a multiple of C)."""
    rng = np.random.default_rng(70 + C)
    d, e, s = 6, 10, 4
    W_u, W_v = rng.normal(size=(d, e)) / 2, rng.normal(size=(d, e)) / 2
    W_z, W_o = rng.normal(size=(d, s)) / 2, rng.normal(size=(e, d)) / 2
    gamma, beta = rng.normal(1.0, 0.3, (4, s)), rng.normal(0.0, 0.3, (4, s))
    relpos = rng.normal(0.0, 0.5, 2 * C - 1)
    X = rng.normal(size=(T, d))
    Tp = -(-T // C) * C
    Xp = np.zeros((1, Tp, d))
    Xp[0, :T] = X
    O, _ = flash_gau(Xp, W_u, W_v, W_z, W_o, gamma, beta, relpos, C, True, lin_scale,
                     local_scale=local_scale)
    st = O_.DecodeState(W_u, W_v, W_z, W_o, gamma, beta, relpos, C, lin_scale, local_scale)
    for t in range(T):
        o = st.step(X[t])
        assert np.allclose(o, O[0, t], rtol=1e-12, atol=1e-12), t


def test_decode_prefix_is_completed_chunks_sum():
    """After k full chunks the linear cache is the sum of their K_lin^T V,
    and the chunk cache is empty."""
    rng = np.random.default_rng(77)
    d, e, s, C = 5, 7, 4, 3
    W = [rng.normal(size=sh) for sh in ((d, e), (d, e), (d, s), (e, d))]
    gamma, beta = rng.normal(1.0, 0.3, (4, s)), rng.normal(0.0, 0.3, (4, s))
    st = O_.DecodeState(*W, gamma, beta, rng.normal(size=2 * C - 1), C)
    X = rng.normal(size=(2 * C, d))
    for x in X:
        st.step(x)
    Z = swish(X @ W[2])
    Kl = Z * gamma[3] + beta[3]
    V = swish(X @ W[1])
    assert np.allclose(st.prefix, Kl.T @ V, rtol=1e-12, atol=1e-12)
    assert st.kq == [] and st.t == 2 * C


# ---------------------------------------------------------------- GlobalOnly
def test_global_only_noncausal_is_full_linear_attention():
    """local_scale = 0, non-causal: only the global term, the total of all
    chunk states, remains; by associativity it is the full-length linear
    attention U * (Q_lin K_lin^T V), computed here with the T x T matrix."""
    rng = np.random.default_rng(80)
    B, T, d, e, s, C = 2, 12, 5, 7, 4, 4
    W_u, W_v = rng.normal(size=(d, e)), rng.normal(size=(d, e))
    W_z, W_o = rng.normal(size=(d, s)), rng.normal(size=(e, d))
    gamma, beta = rng.normal(1, 0.3, (4, s)), rng.normal(0, 0.3, (4, s))
    X = rng.normal(size=(B, T, d))
    O, _ = flash_gau(X, W_u, W_v, W_z, W_o, gamma, beta, rng.normal(size=2 * C - 1), C, False,
                     lin_scale=0.7, local_scale=0.0)
    U, V, Z = swish(X @ W_u), swish(X @ W_v), swish(X @ W_z)
    Ql, Kl = Z * gamma[2] + beta[2], Z * gamma[3] + beta[3]
    want = np.stack([(U[b] * (0.7 * (Ql[b] @ Kl[b].T) @ V[b])) @ W_o for b in range(B)])
    assert np.allclose(O, want, rtol=1e-12, atol=1e-10)


def test_global_only_causal_c1_is_strictly_causal_linear_attention():
    """local_scale = 0, causal, C = 1: token t sees the states of tokens
    t' < t only (a brute-force sum over earlier tokens)."""
    rng = np.random.default_rng(81)
    T, d, e, s = 9, 4, 6, 4
    W_u, W_v = rng.normal(size=(d, e)), rng.normal(size=(d, e))
    W_z, W_o = rng.normal(size=(d, s)), rng.normal(size=(e, d))
    gamma, beta = rng.normal(1, 0.3, (4, s)), rng.normal(0, 0.3, (4, s))
    X = rng.normal(size=(1, T, d))
    O, _ = flash_gau(X, W_u, W_v, W_z, W_o, gamma, beta, np.array([0.3]), 1, True,
                     local_scale=0.0)
    U, V, Z = swish(X[0] @ W_u), swish(X[0] @ W_v), swish(X[0] @ W_z)
    Ql, Kl = Z * gamma[2] + beta[2], Z * gamma[3] + beta[3]
    for t in range(T):
        acc = sum((Ql[t] @ Kl[h]) * V[h] for h in range(t)) if t else np.zeros(e)
        assert np.allclose(O[0, t], (U[t] * acc) @ W_o, rtol=1e-12, atol=1e-12)


def test_output_is_affine_in_local_scale():
    """O(l) = O(0) + l (O(1) - O(0)): the local term enters linearly."""
    rng = np.random.default_rng(82)
    B, T, d, e, s, C = 1, 8, 4, 6, 4, 4
    args = [rng.normal(size=(B, T, d)), rng.normal(size=(d, e)), rng.normal(size=(d, e)),
            rng.normal(size=(d, s)), rng.normal(size=(e, d)), rng.normal(1, 0.3, (4, s)),
            rng.normal(0, 0.3, (4, s)), rng.normal(size=2 * C - 1), C, True]
    O0 = flash_gau(*args, local_scale=0.0)[0]
    O1 = flash_gau(*args, local_scale=1.0)[0]
    O25 = flash_gau(*args, local_scale=2.5)[0]
    assert np.allclose(O25, O0 + 2.5 * (O1 - O0), rtol=1e-12, atol=1e-10)


# ---------------------------------------------------------- segment masks
def _layer_args(rng, B, T, d, e, s, C):
    return dict(X=rng.normal(size=(B, T, d)), W_u=rng.normal(size=(d, e)) / np.sqrt(d),
                W_v=rng.normal(size=(d, e)) / np.sqrt(d), W_z=rng.normal(size=(d, s)) / np.sqrt(d),
                W_o=rng.normal(size=(e, d)) / np.sqrt(e), gamma=rng.normal(1, 0.3, (4, s)),
                beta=rng.normal(0, 0.3, (4, s)), relpos=rng.normal(size=2 * C - 1))


def _call(a, C, causal, **kw):
    return flash_gau(a["X"], a["W_u"], a["W_v"], a["W_z"], a["W_o"], a["gamma"], a["beta"],
                     a["relpos"], C, causal, **kw)[0]


@pytest.mark.parametrize("causal", [True, False])
def test_packed_documents_equal_separate_runs(causal):
    """Two documents packed into one sequence, each a whole number of chunks,
    with one segment id per document: the output on each document's tokens
    equals the layer run on that document alone (the local part never
    crosses a chunk, the masked global part never crosses the boundary)."""
    rng = np.random.default_rng(90)
    d, e, s, C = 6, 8, 4, 4
    a = _layer_args(rng, 1, 5 * C, d, e, s, C)
    seg = np.array([[7, 7, 7, 2, 2]])
    O = _call(a, C, causal, segment_ids=seg)
    for lo, hi in ((0, 3 * C), (3 * C, 5 * C)):
        part = dict(a, X=a["X"][:, lo:hi])
        assert np.allclose(O[:, lo:hi], _call(part, C, causal), rtol=1e-12, atol=1e-12)


def test_one_segment_is_the_unsegmented_layer():
    rng = np.random.default_rng(91)
    a = _layer_args(rng, 2, 12, 5, 6, 4, 3)
    for causal in (True, False):
        O = _call(a, 3, causal, segment_ids=np.full((2, 4), 5))
        assert np.allclose(O, _call(a, 3, causal), rtol=1e-12, atol=1e-12)


def test_distinct_segments_leave_only_the_chunk_itself():
    """Every chunk its own segment: causal, no earlier chunk is visible, so
    the global term vanishes (the LocalOnly output); non-causal, each chunk
    sees exactly itself."""
    rng = np.random.default_rng(92)
    B, T, d, e, s, C = 1, 12, 5, 6, 4, 4
    a = _layer_args(rng, B, T, d, e, s, C)
    seg = np.array([[0, 1, 2]])
    assert np.allclose(_call(a, C, True, segment_ids=seg), _call(a, C, True, lin_scale=0.0),
                       rtol=1e-12, atol=1e-12)
    # non-causal, each chunk alone is the layer run on that chunk
    O = _call(a, C, False, segment_ids=seg)
    for g in range(3):
        part = dict(a, X=a["X"][:, g * C:(g + 1) * C])
        assert np.allclose(O[:, g * C:(g + 1) * C], _call(part, C, False), rtol=1e-12,
                           atol=1e-12)


def test_repeated_id_after_a_gap_starts_a_new_segment():
    """Ids 3, 3, 4, 3: the last chunk is a new run, so causally it sees no
    earlier chunk (the mask row is empty)."""
    M = O.chunk_mask(4, True, [3, 3, 4, 3])
    assert M.tolist() == [[0, 0, 0, 0], [1, 0, 0, 0], [0, 0, 0, 0], [0, 0, 0, 0]]
    M = O.chunk_mask(4, False, [3, 3, 4, 3], average=True)
    assert np.allclose(M, [[.5, .5, 0, 0], [.5, .5, 0, 0], [0, 0, 1, 0], [0, 0, 0, 1]])


def test_chunk_average_matches_token_level_brute_force():
    """Row-normalised mask: the global term of token t is Q_lin,t times the
    mean over the visible chunks of their states, each state summed token by
    token (K_lin,tau^T V_tau) rather than as a matrix product."""
    rng = np.random.default_rng(93)
    B, T, d, e, s, C = 1, 15, 4, 5, 3, 3
    a = _layer_args(rng, B, T, d, e, s, C)
    seg = np.array([[1, 1, 1, 2, 2]])
    for causal in (True, False):
        O_ = _call(a, C, causal, segment_ids=seg, chunk_average=True, local_scale=0.0)
        U = swish(a["X"][0] @ a["W_u"])
        V = swish(a["X"][0] @ a["W_v"])
        Z = swish(a["X"][0] @ a["W_z"])
        Ql, Kl = Z * a["gamma"][2] + a["beta"][2], Z * a["gamma"][3] + a["beta"][3]
        for t in range(T):
            g = t // C
            vis = [h for h in range(5) if seg[0, h] == seg[0, g] and (h < g or not causal)]
            acc = np.zeros(e)
            for h in vis:
                for tau in range(h * C, (h + 1) * C):
                    acc += (Ql[t] @ Kl[tau]) * V[tau]
            if vis:
                acc /= len(vis)
            assert np.allclose(O_[0, t], (U[t] * acc) @ a["W_o"], rtol=1e-12, atol=1e-12)
