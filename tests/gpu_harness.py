"""Shared helpers of the GPU tests: seeded inputs to device tensors, one call
through the C ABI, the oracle on the same inputs, and error measures."""

import numpy as np
import torch

from efficient_attention_transformer_gb300 import binding as bd
from efficient_attention_transformer_gb300.synthetic import make_inputs
from oracle import flash_gau

# Max-abs-error relative to max|reference| (fp32 io: 1e-4, bf16 io: 2e-2).
TOL = {"fp32": 1e-4, "bf16": 2e-2}
# Intermediates are stored in the io type; bf16 storage alone costs up to
# 2^-9 of each element, so they get a tighter bound than the output.
TOL_INTER = {"fp32": 1e-4, "bf16": 1e-2}


def torch_dtype(name):
    return torch.float32 if name == "fp32" else torch.bfloat16


class Case:
    """One problem instance on the GPU plus its float64 oracle result."""

    def __init__(self, B, T, d, e, s, C, causal, dtype, seed, lin_scale=1.0, inputs=None,
                 device="cuda", local_scale=1.0):
        self.B, self.T, self.d, self.e, self.s, self.C = B, T, d, e, s, C
        self.causal, self.dtype, self.lin_scale = causal, dtype, lin_scale
        self.local_scale = local_scale
        self.inp = inputs or make_inputs(B, T, d, e, s, C, dtype, seed)
        tdt = torch_dtype(dtype)
        i = self.inp
        dev = torch.device(device)
        self.X = torch.tensor(i["X"], dtype=tdt, device=dev)
        W_uvz = np.concatenate([i["W_u"], i["W_v"], i["W_z"]], axis=1)
        self.weights = bd.GauWeights(
            torch.tensor(W_uvz, dtype=tdt, device=dev),
            torch.tensor(i["W_o"], dtype=tdt, device=dev),
            torch.tensor(i["gamma"], dtype=torch.float32, device=dev),
            torch.tensor(i["beta"], dtype=torch.float32, device=dev),
            torch.tensor(i["relpos"], dtype=torch.float32, device=dev),
            d, e, s, lin_scale, local_scale)
        self.workspace = self.weights.new_workspace(B, T, C, causal, dev)
        self.out = torch.empty_like(self.X)
        self.layout = bd.workspace_layout(B, T, C, d, e, s, causal, self.weights.dtype)

    def run(self):
        bd.forward(self.X, self.weights, self.C, self.causal, out=self.out,
                   workspace=self.workspace)
        torch.cuda.synchronize()
        return self.out.double().cpu().numpy()

    def reference(self):
        i = self.inp
        return flash_gau(i["X"], i["W_u"], i["W_v"], i["W_z"], i["W_o"], i["gamma"],
                         i["beta"], i["relpos"], self.C, self.causal, self.lin_scale,
                         local_scale=self.local_scale)

    def intermediate(self, name):
        """An intermediate read back from the workspace, as float64, in its
        logical (row-major) shape."""
        tdt = torch_dtype(self.dtype)
        B, T, e, s, M = self.B, self.T, self.e, self.s, self.B * self.T
        G = T // self.C
        shapes = {"U": (M, e), "V": (M, e), "heads": (4, M, s), "gated": (M, e),
                  "state": (B * G, s, e), "prefix": (B * G if self.causal else B, s, e)}
        shape = shapes[name]
        n = int(np.prod(shape))
        raw = self.workspace[self.layout[name]:]
        t = raw[: n * (2 if tdt == torch.bfloat16 else 4)].view(tdt)
        a = t.double().cpu().numpy()
        if tdt == torch.bfloat16 and name in BLOCKED64:
            rows = n // e
            return unblock64(a, rows, e).reshape(shape)
        return a.reshape(shape)

    def status(self):
        return bd.workspace_status(self.workspace)


# bf16 intermediates kept in 64 x 64 blocks, row-block-major (see the
# workspace layout in include/flash_gau.h)
BLOCKED64 = ("V", "state", "prefix")


def unblock64(flat, rows, cols):
    """[rows, cols] from its 64 x 64-blocked storage: block (i, j) is the
    row-major 64 x 64 tile at block index i * (cols / 64) + j."""
    return (flat.reshape(rows // 64, cols // 64, 64, 64).transpose(0, 2, 1, 3)
            .reshape(rows, cols))


def rel_err(got, ref):
    """max|got - ref| / max|ref|."""
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))
