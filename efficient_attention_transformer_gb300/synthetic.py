"""Seeded synthetic inputs for the FLASH GAU forward.

This module only draws random numbers and rounds them to the storage type;
it holds none of the layer's arithmetic.  The tests, the benchmark and the
oracle-side checks all take their inputs from here, so both sides of every
comparison see identical values.

Distributions (fan-in initialisation, per-dimension heads near identity,
small relative-position weights):
  X                ~ N(0, 1)                   [B, T, d]
  W_u, W_v         ~ N(0, variance 1/d)        [d, e]
  W_z              ~ N(0, variance 1/d)        [d, s]
  W_o              ~ N(0, variance 1/e)        [e, d]
  gamma            ~ N(1, std 0.02)            [4, s]  rows Qquad, Kquad, Qlin, Klin
  beta             ~ N(0, std 0.02)            [4, s]
  relpos           ~ N(0, std 0.1)             [2C - 1]
drawn in that order from ``numpy.random.default_rng(seed)`` in float64.
X and the four weight matrices are then rounded to the io type (bf16 by
round-to-nearest-even, or fp32); gamma, beta and relpos are rounded to fp32.
"""

import numpy as np

__all__ = ["WORKLOADS", "workload", "make_inputs", "round_bf16", "round_fp32"]


def _w(B, T, d, e, s, C, causal, dtype, seed):
    return dict(B=B, T=T, d=d, e=e, s=s, C=C, causal=causal, dtype=dtype,
                seed=seed)


# Workloads at the widths the pages use (112M model: d=768, e=2d, s=128;
# ~500M model: d=1024) with chunk sizes 128/256/512 and contexts to 8K.
WORKLOADS = {
    "tiny_causal_fp32_T256": _w(1, 256, 64, 128, 32, 64, True, "fp32", 0),
    "lm112m_causal_B8_T1024": _w(8, 1024, 768, 1536, 128, 256, True, "bf16", 1),
    "mlm112m_noncausal_B32_T512": _w(32, 512, 768, 1536, 128, 256, False, "bf16", 2),
    "long_causal_B2_T8192": _w(2, 8192, 768, 1536, 128, 256, True, "bf16", 3),
    "wide500m_causal_T8192_C128": _w(1, 8192, 1024, 2048, 128, 128, True, "bf16", 4),
    "wide500m_causal_T8192_C256": _w(1, 8192, 1024, 2048, 128, 256, True, "bf16", 4),
    "wide500m_causal_T8192_C512": _w(1, 8192, 1024, 2048, 128, 512, True, "bf16", 4),
    # FLASH-Quad: one chunk spanning the whole sequence (C = T).
    "wide500m_quad_B4_T2048": _w(4, 2048, 1024, 2048, 128, 2048, True, "bf16", 4),
}


def workload(name):
    """A copy of one named workload's shape dictionary."""
    return dict(WORKLOADS[name])


def round_fp32(x):
    """Round float64 values to the nearest float32, returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_bf16(x):
    """Round float64 values to bfloat16 (via float32, nearest-even on the
    upper 16 bits), returned as float64.  Storage conversion only."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def make_inputs(B, T, d, e, s, C, dtype="bf16", seed=0, **_):
    """Draw one seeded input set; every array is float64 holding values
    exactly representable in its storage type."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, T, d))
    W_u = rng.standard_normal((d, e)) / np.sqrt(d)
    W_v = rng.standard_normal((d, e)) / np.sqrt(d)
    W_z = rng.standard_normal((d, s)) / np.sqrt(d)
    W_o = rng.standard_normal((e, d)) / np.sqrt(e)
    gamma = 1.0 + 0.02 * rng.standard_normal((4, s))
    beta = 0.02 * rng.standard_normal((4, s))
    relpos = 0.1 * rng.standard_normal(2 * C - 1)
    io = round_bf16 if dtype == "bf16" else round_fp32
    return dict(X=io(X), W_u=io(W_u), W_v=io(W_v), W_z=io(W_z), W_o=io(W_o),
                gamma=round_fp32(gamma), beta=round_fp32(beta),
                relpos=round_fp32(relpos))
