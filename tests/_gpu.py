"""Running an ``inputgen.Problem`` through the C ABI on the GPU (tests only)."""
from __future__ import annotations

import numpy as np
import torch

import dense_linear_algebra_gb300 as fx


def to_dev(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceProblem:
    """A problem's arrays resident on the GPU."""

    def __init__(self, p, device="cuda"):
        self.p = p
        self.y = to_dev(p.y, device)
        self.v = to_dev(p.v, device)
        self.z = to_dev(p.z, device)
        if p.kind == "dense":
            Xd = to_dev(p.X, device)  # (m, ld)
            if p.x_store == "bf16":  # the values are bfloat16-representable: the conversion is exact
                Xd = Xd.to(torch.bfloat16)
            self.X = Xd[:, : p.n]
        else:
            self.row_ptr = to_dev(p.row_ptr, device)
            self.col_idx = to_dev(p.col_idx, device)
            self.vals = to_dev(p.vals, device)

    def run(self, out=None, stream=None, alpha=None, beta=None):
        p = self.p
        a = p.alpha if alpha is None else alpha
        b = p.beta if beta is None else beta
        if p.kind == "dense":
            return fx.dense(self.X, self.y, self.v, a, b, self.z, out=out, stream=stream)
        return fx.csr(self.row_ptr, self.col_idx, self.vals, self.y, p.n, self.v, a, b, self.z, out=out, stream=stream)


def run_problem(p):
    dp = DeviceProblem(p)
    out = dp.run()
    torch.cuda.synchronize()
    assert fx.device_error() == fx.FXTX_OK
    return out.cpu().numpy().astype(np.float64)
