"""Float64 CPU oracle for the FLASH GAU autoregressive decode step (TEST
INFRASTRUCTURE ONLY: the same import rule as ``oracle.flash_gau``).

[TQLT] §3.2.1 ("Discussion"): decoding takes constant work per token,
O(C d^2), since the global term is carried as one running matrix and the
local attention reaches back within the current chunk only; how that cache
is kept is not stated.  The plainest
reading, written out here for one sequence:

  state     Prefix = sum over completed chunks h of K_lin,h^T V_h  [s, e]
            the current chunk's K_quad, K_lin and V rows so far   [i, *]
  token t   i = t mod C (its place in its chunk)
            u, v, z = swish(x W_u), swish(x W_v), swish(x W_z)
            q_quad, k_quad, q_lin, k_lin = z * gamma_k + beta_k
            append k_quad, k_lin, v to the chunk cache (row i)
            a_j = relu(q_quad . k_quad_j / C + relpos[j - i + C - 1])^2, j <= i
            o = [u * (local_scale sum_j a_j v_j + lin_scale q_lin Prefix)] W_o
  chunk end (i = C - 1): Prefix += K_lin,chunk^T V_chunk; empty the cache

By causality the output for token t equals row t of the forward pass over
the first t + 1 tokens (``flash_gau``, causal); tests/test_oracle.py pins it
there.
"""

import numpy as np

from .flash_gau import scale_offset, swish

__all__ = ["DecodeState"]


class DecodeState:
    """One sequence's decode state (float64)."""

    def __init__(self, W_u, W_v, W_z, W_o, gamma, beta, relpos, C, lin_scale=1.0,
                 local_scale=1.0):
        f = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
        self.W_u, self.W_v, self.W_z, self.W_o = f(W_u), f(W_v), f(W_z), f(W_o)
        self.gamma, self.beta, self.relpos = f(gamma), f(beta), f(relpos)
        self.C, self.lin_scale, self.local_scale = int(C), float(lin_scale), float(local_scale)
        self.e, self.s = self.W_u.shape[1], self.W_z.shape[1]
        self.prefix = np.zeros((self.s, self.e))
        self.kq, self.kl, self.v = [], [], []
        self.t = 0

    def step(self, x):
        """Consumes one token x [d]; returns its output [d]."""
        x = np.asarray(x, dtype=np.float64)
        C = self.C
        i = self.t % C
        u, v, z = swish(x @ self.W_u), swish(x @ self.W_v), swish(x @ self.W_z)
        qq, kq, ql, kl = scale_offset(z, self.gamma, self.beta)
        self.kq.append(kq)
        self.kl.append(kl)
        self.v.append(v)
        K = np.array(self.kq)        # [i + 1, s]
        Vc = np.array(self.v)        # [i + 1, e]
        j = np.arange(i + 1)
        a = np.maximum(K @ qq / C + self.relpos[j - i + C - 1], 0.0) ** 2
        vhat = self.local_scale * (a @ Vc) + self.lin_scale * (ql @ self.prefix)
        o = (u * vhat) @ self.W_o
        if i == C - 1:
            self.prefix = self.prefix + np.array(self.kl).T @ Vc
            self.kq, self.kl, self.v = [], [], []
        self.t += 1
        return o
