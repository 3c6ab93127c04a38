"""Float64 CPU oracle for the FLASH GAU backward pass (TEST INFRASTRUCTURE
ONLY: the same import rule as ``oracle.flash_gau``; the CUDA library never
uses it).

Gradients of the scalar L = sum(dO * O), O = flash_gau(X, ...), with respect
to the input and every parameter of the layer, by the chain rule through the
forward's steps in reverse.  The forward is the one of ``flash_gau`` ([TQLT]
Method, eq. 5, eq. 7, eq. 8 and the display after it); the backward is plain
calculus, written out step by step:

  O = A W_o,  A = U * Vh,  Vh = Vq + Vl
      dW_o = A^T dO,  dA = dO W_o^T,  dU = dA * Vh,  dVh = dA * U
  Vq_g = l P_g V_g,  P = relu(S)^2 (masked),  S = Qq Kq^T / C + b,
  l = local_scale
      dP = l dVh_g V_g^T,  dV_g += l P^T dVh_g,  dS = 2 relu(S) dP (masked)
      dQq_g = dS Kq_g / C,  dKq_g = dS^T Qq_g / C,
      drelpos[j - i + C - 1] += dS[i, j]
  Vl_g = lin_scale Ql_g Prefix_g,  Prefix_g = sum_{h<g} State_h (causal) or
  sum_h State_h,  State_h = Kl_h^T V_h
      dQl_g = lin_scale dVh_g Prefix_g^T,  dPrefix_g = lin_scale Ql_g^T dVh_g
      dState_h = sum_{g>h} dPrefix_g (causal) or sum_g dPrefix_g
      dKl_h = V_h dState_h^T,  dV_h += Kl_h dState_h
  head_k = Z gamma_k + beta_k
      dZ = sum_k dhead_k * gamma_k,  dgamma_k = sum dhead_k * Z,
      dbeta_k = sum dhead_k
  U = swish(X W_u) (V, Z alike), swish'(x) = sig(x) (1 + x (1 - sig(x)))
      dX = sum_w (dU * swish'(X W_u)) W_u^T,  dW_u = X^T (dU * swish'(X W_u))

Pinned by tests/test_oracle.py against central finite differences of L.
"""

import numpy as np

from .flash_gau import relpos_bias, scale_offset, swish

__all__ = ["swish_grad", "flash_gau_backward"]


def swish_grad(x):
    """d/dx of x * sigmoid(x): sigmoid(x) * (1 + x * (1 - sigmoid(x)))."""
    x = np.asarray(x, dtype=np.float64)
    sg = 1.0 / (1.0 + np.exp(-x))
    return sg * (1.0 + x * (1.0 - sg))


def flash_gau_backward(X, W_u, W_v, W_z, W_o, gamma, beta, relpos, C, causal, dO,
                       lin_scale=1.0, local_scale=1.0):
    """Gradients of sum(dO * flash_gau(...)) (same arguments as ``flash_gau``
    without RoPE; dO: [B, T, d]).  Returns a dict with dX [B, T, d], dW_u,
    dW_v [d, e], dW_z [d, s], dW_o [e, d], dgamma, dbeta [4, s] and
    drelpos [2C - 1], all float64."""
    f = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    X, W_u, W_v, W_z, W_o, dO = f(X), f(W_u), f(W_v), f(W_z), f(W_o), f(dO)
    gamma, beta = f(gamma), f(beta)
    B, T, d = X.shape
    if C <= 0 or T % C != 0:
        raise ValueError("T must be a positive multiple of C")
    G = T // C
    e, s = W_u.shape[1], W_z.shape[1]

    # ---- forward, keeping what the backward needs
    Pu, Pv, Pz = X @ W_u, X @ W_v, X @ W_z
    U, V, Z = swish(Pu), swish(Pv), swish(Pz)
    Qq, Kq, Ql, Kl = scale_offset(Z, gamma, beta)
    bias = relpos_bias(relpos, C)
    mask = np.tril(np.ones((C, C))) if causal else np.ones((C, C))
    S = np.zeros((B, G, C, C))
    Vq = np.zeros((B, T, e))
    state = np.zeros((B, G, s, e))
    for b in range(B):
        for g in range(G):
            r = slice(g * C, (g + 1) * C)
            S[b, g] = Qq[b, r] @ Kq[b, r].T / C + bias
            P = np.maximum(S[b, g], 0.0) ** 2 * mask
            Vq[b, r] = local_scale * (P @ V[b, r])
            state[b, g] = Kl[b, r].T @ V[b, r]
    prefix = np.zeros((B, G, s, e))
    for b in range(B):
        for g in range(G):
            prefix[b, g] = state[b, :g].sum(axis=0) if causal else state[b].sum(axis=0)
    Vl = np.zeros((B, T, e))
    for b in range(B):
        for g in range(G):
            r = slice(g * C, (g + 1) * C)
            Vl[b, r] = lin_scale * (Ql[b, r] @ prefix[b, g])
    Vh = Vq + Vl
    A = U * Vh

    # ---- output projection and gate
    dW_o = np.einsum("bte,btd->ed", A, dO)
    dA = dO @ W_o.T
    dU = dA * Vh
    dVh = dA * U

    # ---- local (quadratic) part, chunk by chunk
    dV = np.zeros((B, T, e))
    dQq, dKq = np.zeros((B, T, s)), np.zeros((B, T, s))
    drelpos = np.zeros(2 * C - 1)
    ii, jj = np.meshgrid(np.arange(C), np.arange(C), indexing="ij")
    for b in range(B):
        for g in range(G):
            r = slice(g * C, (g + 1) * C)
            relu = np.maximum(S[b, g], 0.0)
            P = relu ** 2 * mask
            dP = local_scale * (dVh[b, r] @ V[b, r].T)
            dV[b, r] += local_scale * (P.T @ dVh[b, r])
            dS = 2.0 * relu * dP * mask
            dQq[b, r] = dS @ Kq[b, r] / C
            dKq[b, r] = dS.T @ Qq[b, r] / C
            np.add.at(drelpos, (jj - ii + C - 1).ravel(), dS.ravel())

    # ---- global (linear) part
    dQl, dKl = np.zeros((B, T, s)), np.zeros((B, T, s))
    dprefix = np.zeros((B, G, s, e))
    for b in range(B):
        for g in range(G):
            r = slice(g * C, (g + 1) * C)
            dQl[b, r] = lin_scale * (dVh[b, r] @ prefix[b, g].T)
            dprefix[b, g] = lin_scale * (Ql[b, r].T @ dVh[b, r])
    for b in range(B):
        for h in range(G):
            dstate = dprefix[b, h + 1:].sum(axis=0) if causal else dprefix[b].sum(axis=0)
            r = slice(h * C, (h + 1) * C)
            dKl[b, r] = V[b, r] @ dstate.T
            dV[b, r] += Kl[b, r] @ dstate

    # ---- the four heads
    dH = np.stack([dQq, dKq, dQl, dKl])  # [4, B, T, s]
    dZ = np.einsum("kbts,ks->bts", dH, gamma)
    dgamma = np.einsum("kbts,bts->ks", dH, Z)
    dbeta = dH.sum(axis=(1, 2))

    # ---- projections through swish
    dPu, dPv, dPz = dU * swish_grad(Pu), dV * swish_grad(Pv), dZ * swish_grad(Pz)
    dX = dPu @ W_u.T + dPv @ W_v.T + dPz @ W_z.T
    dW_u = np.einsum("btd,bte->de", X, dPu)
    dW_v = np.einsum("btd,bte->de", X, dPv)
    dW_z = np.einsum("btd,bts->ds", X, dPz)
    return dict(dX=dX, dW_u=dW_u, dW_v=dW_v, dW_z=dW_z, dW_o=dW_o, dgamma=dgamma,
                dbeta=dbeta, drelpos=drelpos)
