"""Float64 CPU oracle for the FLASH gated-attention-unit forward pass with
mixed chunk attention.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plainly written
definition that the CUDA path is checked against.  Only the test suite, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py``
may import it; the library itself never does, and it shares no code with the
CUDA kernels.

Sources ("the pages"):
  [FLASH-blog]  "FLASH: Possibly the Most Interesting Efficient Transformer
                Design in Recent Times" (kexue.fm, translated), sections
                "Gated Attention", "Weak Attention", "Mixed Chunking".
  [TQLT]        "Transformer Quality in Linear Time" (wikillm summary of
                arXiv 2202.10447): Method, eq. 5, eq. 7, eq. 8, and the
                gau_block / flash_block pseudocode.
  [TQLT-zh]     "Transformer Quality in Linear Time" (papercache summary),
                appendix D, Code 4 (relative position bias).

Readings taken where the pages disagree or are silent:
  * scores are scaled by 1/C inside relu^2, before the bias is added
    ([TQLT] flash_block pseudocode; gau_block divides by the length N, which
    is the same rule at C = T);
  * the global term is the plain sum of chunk states of eq. 7 / eq. 8, times
    a caller-chosen ``lin_scale`` (1 = eq. 7/8, 1/C = the listing's division,
    0 = the LocalOnly ablation); the local term is likewise multiplied by
    ``local_scale`` (1 = as written, 0 = the GlobalOnly ablation of [TQLT]
    §4.4, which keeps only the global part);
  * b[i, j] = relpos[j - i + C - 1], the Toeplitz matrix the Code 4 listing
    builds from 2C-1 weights, used for every C;
  * the causal mask keeps the diagonal (j <= i) and is applied after relu^2;
  * the causal global term of the first chunk is the empty sum, i.e. zero;
  * segment masks (packed text) act on the global term only, at chunk
    granularity: a segment is a maximal run of consecutive chunks with one
    id, and the optional row normalisation makes the global term the mean
    of the visible chunk states (``chunk_mask``);
  * no bias terms, norm, RoPE or residual in ``flash_gau`` (the layer as
    eq. 3-8 write it); ``flash_block`` adds the pre-norm, RoPE on the four
    heads over global token positions and the residual of the pages'
    flash_block, with these readings of what the pages leave unprinted:
    the norm is LayerNorm (mean / biased variance, eps inside the square
    root, learned scale and shift) or ScaleNorm (g * x / ||x||), the two the
    pages name; RoPE rotates consecutive pairs (h_2i, h_2i+1) of each head by
    the angle p * base^(-2i/s), p the token's position in its sequence (plus
    an optional offset), base 10000 by default (the rotary embedding as its
    author defines it; the pages print no rope function).

Parity: every function here is pinned by tests/test_oracle.py against
independent formulations (a scalar token loop, the full-length linear
attention of the pages' associativity argument, a library Toeplitz
constructor, the GLU special case, chunk-permutation invariance, golden
fixtures derived by hand from the Code 4 listing).
"""

import numpy as np

__all__ = [
    "swish",
    "scale_offset",
    "relpos_bias",
    "chunk_scores",
    "layer_norm",
    "scale_norm",
    "rope",
    "rope_toeplitz_bias",
    "toeplitz_relpos",
    "flash_gau",
    "flash_block",
    "algorithmic_flops_per_token",
]


def swish(x):
    """SiLU / Swish, phi(x) = x * sigmoid(x) = x / (1 + exp(-x)).

    [FLASH-blog] "Gated Attention": the paper applies Swish to U and V (and
    [TQLT] gau_block applies it to the whole 2e+s projection, so to Z too).
    Written as x / (1 + exp(-x)); for very negative x, exp(-x) overflows to
    inf and the quotient is the correct limit -0.0.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def scale_offset(Z, gamma, beta):
    """The four per-dimension affine heads of mixed chunk attention.

    [TQLT] Method: queries and keys come from Z by a per-dimension scale and
    offset; FLASH derives four heads Q_quad, K_quad, Q_lin, K_lin from the
    same Z ([TQLT] "Mixed chunk attention"; [FLASH-blog] "Mixed Chunking").

    Z: [..., s];  gamma, beta: [4, s] with rows (Q_quad, K_quad, Q_lin, K_lin).
    Returns a tuple of four arrays shaped like Z.
    """
    Z = np.asarray(Z, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    return tuple(Z * gamma[h] + beta[h] for h in range(4))


def relpos_bias(relpos, n):
    """Relative position bias for one length-n window: a Toeplitz matrix
    built from 2n-1 learned weights, b[i, j] = relpos[j - i + n - 1].

    [TQLT-zh] appendix D, Code 4 (the n < 512 branch): the listing pads,
    tiles, reshapes and slices the weight vector; worked by hand for n = 3
    that yields row i = (w[2-i], w[3-i], w[4-i]), i.e. the index rule above
    (tests/golden/relpos_toeplitz_n3.txt).
    """
    relpos = np.asarray(relpos, dtype=np.float64)
    if relpos.shape != (2 * n - 1,):
        raise ValueError("relpos must have 2n-1 entries")
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return relpos[j - i + n - 1]


def chunk_scores(q, k, bias, C, causal):
    """Attention weights inside one chunk: A = relu^2(q k^T / C + b), with
    entries above the diagonal set to zero when causal.

    [TQLT] eq. 5 (relu^2 of scores plus relative bias) and the flash_block
    pseudocode (division by C before the bias, lower-triangular mask applied
    to the relu^2 kernel); [FLASH-blog] "Mixed Chunking" (decoders mask out
    the upper triangle).
    """
    s = q @ k.T / C + bias
    a = np.maximum(s, 0.0) ** 2
    if causal:
        a = np.tril(a)  # keeps j <= i
    return a


def layer_norm(x, g, b, eps=1e-5):
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * g + b,
    var the biased (1/d) variance.  One of the two pre-norms the pages name
    ([TQLT] gau_block / flash_block pseudocode "norm(x)"; [TQLT-zh]
    appendix B.2 and D, Code 5, whose body the page does not print)."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(g, dtype=np.float64) + \
        np.asarray(b, dtype=np.float64)


def scale_norm(x, g, eps=1e-5):
    """ScaleNorm over the last axis: g * x / max(||x||_2, eps), with a single
    learned scalar g ([TQLT-zh] appendix B.2: ScaleNorm in some masked-LM
    models, as a faster stand-in for LayerNorm)."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    return float(g) * x / np.maximum(n, eps)


def rope(h, positions, base=10000.0):
    """Rotary position embedding of the last axis (s even): the pair
    (h[2i], h[2i+1]) of the vector at position p is rotated by the angle
    p * base^(-2i/s).  [TQLT] flash_block pseudocode: RoPE on the four heads,
    with positions counted along the whole sequence rather than from the
    start of each chunk; [FLASH-blog]: the models use RoPE.

    h: [..., T, s]; positions: [T] (one position per row of h)."""
    h = np.asarray(h, dtype=np.float64)
    s = h.shape[-1]
    if s % 2:
        raise ValueError("RoPE needs an even head width")
    inv_freq = float(base) ** (-2.0 * np.arange(s // 2) / s)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos, sin = np.cos(ang), np.sin(ang)
    even, odd = h[..., 0::2], h[..., 1::2]
    out = np.empty_like(h)
    out[..., 0::2] = even * cos - odd * sin
    out[..., 1::2] = even * sin + odd * cos
    return out


def rope_toeplitz_bias(a, b, n, base=10000.0):
    """Relative position bias of a length-n window built from two learned
    vectors with RoPE: [TQLT-zh] appendix D, Code 4, the branch for windows
    of 512 positions and more.  Both vectors are tiled over the n positions,
    each copy rotated by RoPE at its row's position, and the bias is the
    n x n matrix of their dot products: bias[i, j] = rope(a)_i . rope(b)_j.

    a, b: [m], m even (the listing uses m = 128).  Same rotary convention as
    ``rope`` (consecutive pairs, angle p * base^(-2i/m))."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape or a.ndim != 1:
        raise ValueError("a and b must be vectors of the same length")
    pos = np.arange(n)
    A = rope(np.tile(a[None, :], (n, 1)), pos, base)
    Bm = rope(np.tile(b[None, :], (n, 1)), pos, base)
    return A @ Bm.T


def toeplitz_relpos(T):
    """The 2n-1 weights of an n x n Toeplitz matrix in the layer's table
    form, relpos[j - i + n - 1] = T[i, j]: offsets j - i < 0 read down the
    first column, offsets >= 0 along the first row.  The inverse of
    ``relpos_bias``."""
    T = np.asarray(T, dtype=np.float64)
    n = T.shape[0]
    out = np.empty(2 * n - 1)
    for k in range(2 * n - 1):
        d = k - (n - 1)
        out[k] = T[0, d] if d >= 0 else T[-d, 0]
    return out


def chunk_mask(G, causal, segment_ids=None, average=False):
    """The G x G chunk mask of the global term ([TQLT] Paper vs code, the
    segment-mask item: a chunk mask built from segment ids, applied to the
    chunk summaries in the linear part only, each row optionally normalised
    to sum to one with empty rows left at zero).

    M[g, h] = 1 when chunk g sees chunk h: h < g if causal (eq. 8), every h
    otherwise (eq. 7), and g and h lie in one segment.  Reading: a segment
    is a maximal run of consecutive chunks with equal id (packed text puts
    each document in one run); segment_ids=None is one segment.  With
    ``average`` each non-empty row is divided by its number of ones, so the
    global term becomes the mean of the visible chunk states."""
    M = np.zeros((G, G))
    for g in range(G):
        for h in range(G):
            if causal and h >= g:
                continue
            if segment_ids is not None:
                lo, hi = min(g, h), max(g, h)
                if any(segment_ids[k] != segment_ids[g] for k in range(lo, hi + 1)):
                    continue
            M[g, h] = 1.0
    if average:
        n = M.sum(axis=1, keepdims=True)
        M = np.divide(M, n, out=np.zeros_like(M), where=n > 0)
    return M


def flash_gau(X, W_u, W_v, W_z, W_o, gamma, beta, relpos, C, causal,
              lin_scale=1.0, positions=None, rope_base=10000.0, local_scale=1.0,
              segment_ids=None, chunk_average=False):
    """FLASH GAU layer forward with mixed chunk attention, in float64.

    Steps ([TQLT] Method and flash_block; [FLASH-blog] "Mixed Chunking"):
      1. U = swish(X W_u), V = swish(X W_v), Z = swish(X W_z).
      2. Q_quad, K_quad, Q_lin, K_lin = Z * gamma_h + beta_h.
      3. Per chunk g of C tokens: Vq_g = local_scale *
         relu^2(Q_quad,g K_quad,g^T / C + b) V_g (upper triangle zeroed when
         causal).
      4. State_g = K_lin,g^T V_g.
      5. Prefix_g = sum_{h<g} State_h if causal (eq. 8), else sum_h State_h
         (eq. 7).
      6. Vl_g = lin_scale * Q_lin,g Prefix_g.
      7. O_g = [U_g * (Vq_g + Vl_g)] W_o   ([TQLT] display after eq. 8).

    X: [B, T, d]; W_u, W_v: [d, e]; W_z: [d, s]; W_o: [e, d];
    gamma, beta: [4, s]; relpos: [2C-1]; T must be a multiple of C
    ([FLASH-blog] "Mixed Chunking" assumes divisibility).  With
    ``positions`` ([T]) the four heads are rotated by ``rope`` after step 2
    (the flash_block reading); the default keeps eq. 3-8 as written.
    With ``segment_ids`` ([B, G] chunk ids) or ``chunk_average``, step 5
    weighs the states by ``chunk_mask``: Prefix_g = sum_h M[g, h] State_h.

    Returns (O, inter) with O: [B, T, d] float64 and ``inter`` a dict of the
    intermediates U, V, Z, heads [4, B, T, s], state [B, G, s, e],
    prefix [B, G, s, e], Vq, Vl, gated [B, T, e].
    """
    X = np.asarray(X, dtype=np.float64)
    B, T, d = X.shape
    if C <= 0 or T % C != 0:
        raise ValueError("T must be a positive multiple of C")
    G = T // C
    e = W_u.shape[1]
    s = W_z.shape[1]

    U = swish(X @ np.asarray(W_u, dtype=np.float64))
    V = swish(X @ np.asarray(W_v, dtype=np.float64))
    Z = swish(X @ np.asarray(W_z, dtype=np.float64))
    Qq, Kq, Ql, Kl = scale_offset(Z, gamma, beta)
    if positions is not None:
        Qq, Kq, Ql, Kl = (rope(h, positions, rope_base) for h in (Qq, Kq, Ql, Kl))
    bias = relpos_bias(relpos, C)

    Vq = np.zeros((B, T, e))
    state = np.zeros((B, G, s, e))
    for b in range(B):
        for g in range(G):
            rows = slice(g * C, (g + 1) * C)
            a = chunk_scores(Qq[b, rows], Kq[b, rows], bias, C, causal)
            Vq[b, rows] = local_scale * (a @ V[b, rows])
            state[b, g] = Kl[b, rows].T @ V[b, rows]

    prefix = np.zeros((B, G, s, e))
    if segment_ids is None and not chunk_average:
        for b in range(B):
            total = np.zeros((s, e))
            for g in range(G):
                if causal:
                    prefix[b, g] = total  # strictly earlier chunks only
                total = total + state[b, g]
            if not causal:
                prefix[b, :] = total
    else:
        for b in range(B):
            seg = None if segment_ids is None else np.asarray(segment_ids)[b]
            M = chunk_mask(G, causal, seg, chunk_average)
            for g in range(G):
                for h in range(G):
                    if M[g, h] != 0.0:
                        prefix[b, g] += M[g, h] * state[b, h]

    Vl = np.zeros((B, T, e))
    for b in range(B):
        for g in range(G):
            rows = slice(g * C, (g + 1) * C)
            Vl[b, rows] = lin_scale * (Ql[b, rows] @ prefix[b, g])

    gated = U * (Vq + Vl)
    O = gated @ np.asarray(W_o, dtype=np.float64)
    inter = dict(U=U, V=V, Z=Z, heads=np.stack([Qq, Kq, Ql, Kl]),
                 state=state, prefix=prefix, Vq=Vq, Vl=Vl, gated=gated)
    return O, inter


def flash_block(X, W_u, W_v, W_z, W_o, gamma, beta, relpos, C, causal,
                lin_scale=1.0, norm="layer", norm_g=None, norm_b=None, norm_eps=1e-5,
                local_scale=1.0,
                rope_on=True, rope_base=10000.0, pos_offset=0):
    """The pages' FLASH block around the layer ([TQLT] flash_block
    pseudocode): shortcut = x; x = norm(x); the GAU of ``flash_gau`` with
    RoPE on its four heads at the tokens' global positions (t + pos_offset
    for token t of a sequence); return out + shortcut.

    norm: "layer" (``layer_norm`` with norm_g, norm_b [d]), "scale"
    (``scale_norm`` with the scalar norm_g) or None.  Returns (Y, inter)
    with inter from ``flash_gau`` plus Xn, the normalised input."""
    X = np.asarray(X, dtype=np.float64)
    if norm == "layer":
        Xn = layer_norm(X, norm_g, norm_b, norm_eps)
    elif norm == "scale":
        Xn = scale_norm(X, norm_g, norm_eps)
    elif norm is None:
        Xn = X
    else:
        raise ValueError("norm must be 'layer', 'scale' or None")
    T = X.shape[1]
    positions = np.arange(T) + pos_offset if rope_on else None
    O, inter = flash_gau(Xn, W_u, W_v, W_z, W_o, gamma, beta, relpos, C, causal,
                         lin_scale, positions=positions, rope_base=rope_base,
                         local_scale=local_scale)
    inter["Xn"] = Xn
    return O + X, inter


def algorithmic_flops_per_token(d, e, s, C, causal, quad_only=False):
    """Floating-point operations the layer must do per token (one multiply
    plus one add counted as two), excluding the masked upper triangle:

      projection 2d(2e+s) + output 2ed + scores 2*Cbar*s + mixing 2*Cbar*e
      + chunk state 2se + linear read-out 2se,

    with Cbar = (C+1)/2 when causal (average visible keys per query) and C
    otherwise; the two linear-term products are omitted for FLASH-Quad
    (C = T, causal, no global term).
    """
    cbar = (C + 1) / 2.0 if causal else float(C)
    f = 2 * d * (2 * e + s) + 2 * e * d + 2 * cbar * s + 2 * cbar * e
    if not quad_only:
        f += 4 * s * e
    return f
