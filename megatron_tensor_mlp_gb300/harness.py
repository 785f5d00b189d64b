"""Device buffers for one MLP workload (PyTorch provides memory and streams).

Inputs come from the seeded generator in their unsharded layout, are copied to
the device, and are brought to the shard layout by the library's own layout
kernel (``tpmlp_shard_columns``).  All computation goes through the C-ABI.
"""
from __future__ import annotations

import numpy as np
import torch

from . import synth
from . import tpmlp as T


def to_torch(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Host array (bf16 as uint16 patterns, or fp32) -> device tensor of the same bytes."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> fp64 numpy array of its exact values."""
    return t.detach().float().cpu().numpy().astype(np.float64)


class MLPBuffers:
    """All tensors of one forward (+ backward) pass of a workload on one device."""

    def __init__(self, wl: synth.Workload, device="cuda", backward=None, host=None, grad_f32=True):
        self.wl = wl
        self.device = device
        bwd = wl.backward if backward is None else backward
        M, h, f, p = wl.M, wl.h, wl.ffn, wl.p
        fs = f // p
        self.dt = T.F32 if wl.dtype == "f32" else T.BF16
        tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        gdt = torch.float32 if (grad_f32 or wl.dtype == "f32") else torch.bfloat16
        self.grad_dt = T.F32 if gdt == torch.float32 else T.BF16
        host = host if host is not None else {k: wl.gen(k) for k in ("X", "A", "B", "b1", "b2")}
        if bwd and "dZ" not in host:
            host["dZ"] = wl.gen("dZ")
        self.host = host
        self.X = to_torch(host["X"], device)
        A = to_torch(host["A"], device)
        self.A_sh = torch.empty((p, h, fs), dtype=tdt, device=device)
        T.tpmlp_shard_columns(A, self.A_sh, h, f, p, self.dt)
        del A
        # B [f, h] row-major already is [p][fs][h]; b1 [f] already is [p][fs]
        self.B_sh = to_torch(host["B"], device).view(p, fs, h)
        self.b1_sh = None if host["b1"] is None else to_torch(host["b1"], device).view(p, fs)
        self.b2 = None if host["b2"] is None else to_torch(host["b2"], device)
        self.Z = torch.empty((M, h), dtype=tdt, device=device)
        self.Y = torch.empty((p, M, fs), dtype=tdt, device=device)
        self.H = torch.empty((p, M, fs), dtype=tdt, device=device) if bwd else None
        self.backward = bwd
        if bwd:
            self.dZ = to_torch(host["dZ"], device)
            self.dX = torch.empty((M, h), dtype=tdt, device=device)
            self.dA_sh = torch.empty((p, h, fs), dtype=gdt, device=device)
            self.dB_sh = torch.empty((p, fs, h), dtype=gdt, device=device)
            self.db1_sh = torch.empty((p, fs), dtype=gdt, device=device)
            self.db2 = torch.empty((h,), dtype=gdt, device=device)
            self.dH = torch.empty((p, M, fs), dtype=tdt, device=device)

    def dims(self):
        w = self.wl
        return w.s, w.b, w.h, w.ffn, w.p

    def fwd(self, stream=None):
        T.tpmlp_mlp_fwd(self.X, self.A_sh, self.b1_sh, self.B_sh, self.b2, self.Z, self.Y, self.H, *self.dims(),
                        dt=self.dt, stream=stream)

    def bwd(self, stream=None):
        T.tpmlp_mlp_bwd(self.X, self.A_sh, self.B_sh, self.H, self.Y, self.dZ, self.dX, self.dA_sh, self.dB_sh,
                        self.db1_sh, self.db2, self.dH, *self.dims(), dt=self.dt, grad_dt=self.grad_dt, stream=stream)

    # unsharded views of the sharded results (for comparisons)
    def Y_full(self):
        p, M, fs = self.Y.shape
        return self.Y.permute(1, 0, 2).reshape(M, p * fs)

    def H_full(self):
        p, M, fs = self.H.shape
        return self.H.permute(1, 0, 2).reshape(M, p * fs)

    def dA_full(self):
        p, h, fs = self.dA_sh.shape
        return self.dA_sh.permute(1, 0, 2).reshape(h, p * fs)

    def dB_full(self):
        p, fs, h = self.dB_sh.shape
        return self.dB_sh.reshape(p * fs, h)
