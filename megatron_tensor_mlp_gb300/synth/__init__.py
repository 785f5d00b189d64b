"""Seeded synthetic inputs (shared by tests, the benchmark and the oracle checks).

Holds no arithmetic of the MLP: it draws normals with a counter-based
generator (see ``synth.c`` for its definition), stores them in the tensors'
storage type (bf16 bit patterns or fp32), widens bf16 exactly to fp64 and
names the five benchmark workloads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libtpmlp_synth.so")
_lib = None

# tensor stream ids
STREAM_X, STREAM_A, STREAM_B, STREAM_B1, STREAM_B2, STREAM_DZ = 1, 2, 3, 4, 5, 6


def build(force: bool = False) -> str:
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, d, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, d, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, d, vp]
        lib.synth_bf16_to_f64.argtypes = [vp, i64, vp]
        _lib = lib
    return _lib


def normal(seed: int, stream: int, shape, sigma: float, dtype: str = "bf16", offset: int = 0) -> np.ndarray:
    """sigma * N(0,1) draws.  dtype 'bf16' returns uint16 bit patterns, 'f32' float32."""
    n = int(np.prod(shape)) if len(shape) else 1
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        _load().synth_normal_bf16(seed, stream, offset, n, float(sigma), out.ctypes.data)
    elif dtype == "f32":
        out = np.empty(n, dtype=np.float32)
        _load().synth_normal_f32(seed, stream, offset, n, float(sigma), out.ctypes.data)
    else:
        raise ValueError(dtype)
    return out.reshape(shape)


def widen(a: np.ndarray) -> np.ndarray:
    """Exact fp64 values of a bf16 (uint16 patterns) or fp32 array."""
    if a.dtype == np.uint16:
        a = np.ascontiguousarray(a)
        out = np.empty(a.shape, dtype=np.float64)
        _load().synth_bf16_to_f64(a.ctypes.data, a.size, out.ctypes.data)
        return out
    return np.asarray(a, dtype=np.float64)


@dataclass(frozen=True)
class Workload:
    """One benchmark / parity workload: shapes and input distributions."""
    name: str
    s: int
    b: int
    h: int
    ffn: int
    p: int
    dtype: str            # 'f32' or 'bf16'
    sigma_x: float
    sigma_w: float        # A and B
    sigma_bias: float     # 0 -> no bias tensors
    backward: bool
    seed: int

    @property
    def M(self) -> int:
        return self.s * self.b

    def fwd_flops(self) -> float:
        return 4.0 * self.M * self.h * self.ffn

    def bwd_flops(self) -> float:
        return 8.0 * self.M * self.h * self.ffn

    def gen(self, what: str, offset_rows: int = 0, rows: int | None = None):
        """Generate one tensor of the workload (unsharded layout).

        what: 'X' [M,h], 'A' [h,f], 'B' [f,h], 'b1' [f], 'b2' [h], 'dZ' [M,h].
        offset_rows/rows select a row window of X or dZ (same values as the full tensor).
        """
        M, h, f = self.M, self.h, self.ffn
        if what in ("X", "dZ"):
            r = M - offset_rows if rows is None else rows
            stream = STREAM_X if what == "X" else STREAM_DZ
            return normal(self.seed, stream, (r, h), self.sigma_x, self.dtype, offset=offset_rows * h)
        if what == "A":
            return normal(self.seed, STREAM_A, (h, f), self.sigma_w, self.dtype)
        if what == "B":
            return normal(self.seed, STREAM_B, (f, h), self.sigma_w, self.dtype)
        if what == "b1":
            return normal(self.seed, STREAM_B1, (f,), self.sigma_bias, self.dtype) if self.sigma_bias > 0 else None
        if what == "b2":
            return normal(self.seed, STREAM_B2, (h,), self.sigma_bias, self.dtype) if self.sigma_bias > 0 else None
        raise ValueError(what)


# The five workloads: shapes [s,b,h], FFN width, shard count and distributions.
WORKLOADS = {
    1: Workload("tiny-f32-fwd-bwd s8 b2 h64 ffn256 p2", 8, 2, 64, 256, 2, "f32", 1.0, 0.02, 0.0, True, 0),
    2: Workload("bf16-fwd s512 b4 h1024 ffn4096 p4", 512, 4, 1024, 4096, 4, "bf16", 1.0, 0.02, 0.01, False, 1),
    3: Workload("bf16-fwd s2048 b2 h4096 ffn16384 p8", 2048, 2, 4096, 16384, 8, "bf16", 1.0, 0.02, 0.0, False, 2),
    4: Workload("bf16-fwd s4096 b1 h8192 ffn32768 p8", 4096, 1, 8192, 32768, 8, "bf16", 1.0, 0.01, 0.0, False, 3),
    5: Workload("bf16-fwd-bwd s2048 b4 h5120 ffn20480 p4", 2048, 4, 5120, 20480, 4, "bf16", 1.0, 0.02, 0.0, True, 4),
}


def custom(s, b, h, ffn, p, dtype="bf16", sigma_w=0.02, sigma_bias=0.01, seed=17, backward=True) -> Workload:
    """A small ad-hoc workload (ragged tails, odd shard counts) with the same recipe."""
    return Workload(f"custom s{s} b{b} h{h} ffn{ffn} p{p} {dtype}", s, b, h, ffn, p, dtype,
                    1.0, sigma_w, sigma_bias, backward, seed)
