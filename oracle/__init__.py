"""ORACLE - test infrastructure only.

ctypes wrapper around ``tpmlp_oracle.c``: a plain fp64 CPU statement of the
Megatron tensor-parallel MLP block (column-parallel GeLU(X A), row-parallel
Y B, summed over shards) and its gradients, written as the unsharded
definition.  The header of ``tpmlp_oracle.c`` names the passages it follows.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It imports nothing from the CUDA package.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "tpmlp_oracle.c")
_SO = os.path.join(_HERE, "libtpmlp_oracle.so")

ACT_NONE, ACT_GELU, ACT_RELU = 0, 1, 2

GCC_FLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file to a shared library (fp64, no FMA contraction)."""
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out) or ".")
    os.close(fd)
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(SRC):
        return _SO
    return compile_source(SRC, _SO)


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """One loaded build of the oracle library."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        d, i64, i32, vp = ctypes.c_double, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_gelu.restype = d
        lib.oracle_gelu.argtypes = [d]
        lib.oracle_gelu_grad.restype = d
        lib.oracle_gelu_grad.argtypes = [d]
        lib.oracle_num_threads.restype = i32
        lib.oracle_mlp_fwd.restype = None
        lib.oracle_mlp_fwd.argtypes = [i64, i64, i64, i32] + [vp] * 8
        lib.oracle_mlp_bwd.restype = None
        lib.oracle_mlp_bwd.argtypes = [i64, i64, i64, i32] + [vp] * 12
        lib.oracle_bwd_dX_rows.restype = None
        lib.oracle_bwd_dX_rows.argtypes = [i64, i64, i64, i32] + [vp] * 5 + [i64, vp, vp]
        lib.oracle_bwd_ffn_cols.restype = None
        lib.oracle_bwd_ffn_cols.argtypes = [i64, i64, i64, i32] + [vp] * 5 + [i64, vp, vp, vp, vp]
        lib.oracle_linear_fwd.restype = None
        lib.oracle_linear_fwd.argtypes = [i64, i64, i64, vp, vp, vp, vp]
        lib.oracle_linear_bwd.restype = None
        lib.oracle_linear_bwd.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp]
        lib.oracle_silu.restype = d
        lib.oracle_silu.argtypes = [d]
        lib.oracle_silu_grad.restype = d
        lib.oracle_silu_grad.argtypes = [d]
        lib.oracle_swiglu_fwd.restype = None
        lib.oracle_swiglu_fwd.argtypes = [i64, i64, i64] + [vp] * 11
        lib.oracle_swiglu_bwd.restype = None
        lib.oracle_swiglu_bwd.argtypes = [i64, i64, i64] + [vp] * 16
        lib.oracle_swiglu_pack.restype = None
        lib.oracle_swiglu_pack.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp]
        lib.oracle_bwd_db2.restype = None
        lib.oracle_bwd_db2.argtypes = [i64, i64, vp, vp]
        lib.oracle_shard_columns.restype = None
        lib.oracle_shard_columns.argtypes = [i64, i64, i64, i64, vp, vp]
        lib.oracle_qkv_src_col.restype = i64
        lib.oracle_qkv_src_col.argtypes = [i64, i64, i64]
        lib.oracle_qkv_interleave.restype = None
        lib.oracle_qkv_interleave.argtypes = [i64, i64, i64, i64, i32, vp, vp]
        self.lib = lib
        self.path = so_path

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def gelu(self, z: float) -> float:
        return float(self.lib.oracle_gelu(float(z)))

    def gelu_grad(self, z: float) -> float:
        return float(self.lib.oracle_gelu_grad(float(z)))

    def mlp_fwd(self, X, A, b1, B, b2, act=ACT_GELU):
        """Unsharded forward. X [M,h], A [h,f], B [f,h]; returns (H, Y, Z) in fp64."""
        X, A, B, b1, b2 = _f64(X), _f64(A), _f64(B), _f64(b1), _f64(b2)
        M, h = X.shape
        f = A.shape[1]
        assert A.shape == (h, f) and B.shape == (f, h)
        H = np.empty((M, f)); Y = np.empty((M, f)); Z = np.empty((M, h))
        self.lib.oracle_mlp_fwd(M, h, f, act, _ptr(X), _ptr(A), _ptr(b1), _ptr(B), _ptr(b2),
                                _ptr(H), _ptr(Y), _ptr(Z))
        return H, Y, Z

    def mlp_bwd(self, X, A, B, H, Y, dZ, act=ACT_GELU, with_bias_grads=True):
        """Unsharded backward. Returns dict dX, dA, dB, db1, db2 in fp64."""
        X, A, B, H, Y, dZ = map(_f64, (X, A, B, H, Y, dZ))
        M, h = X.shape
        f = A.shape[1]
        dX = np.empty((M, h)); dA = np.empty((h, f)); dB = np.empty((f, h))
        db1 = np.empty(f) if with_bias_grads else None
        db2 = np.empty(h) if with_bias_grads else None
        work = np.empty((M, f))
        self.lib.oracle_mlp_bwd(M, h, f, act, _ptr(X), _ptr(A), _ptr(B), _ptr(H), _ptr(Y), _ptr(dZ),
                                _ptr(dX), _ptr(dA), _ptr(dB), _ptr(db1), _ptr(db2), _ptr(work))
        return {"dX": dX, "dA": dA, "dB": dB, "db1": db1, "db2": db2}

    def bwd_dX_rows(self, X, A, b1, B, dZ, rows, act=ACT_GELU):
        """dX[rows, :] element by element."""
        X, A, b1, B, dZ = map(_f64, (X, A, b1, B, dZ))
        M, h = X.shape
        f = A.shape[1]
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((len(rows), h))
        self.lib.oracle_bwd_dX_rows(M, h, f, act, _ptr(X), _ptr(A), _ptr(b1), _ptr(B), _ptr(dZ),
                                    len(rows), _ptr(rows), _ptr(out))
        return out

    def bwd_ffn_cols(self, X, A, b1, B, dZ, cols, act=ACT_GELU):
        """Returns (dA[:, cols] as [h, n], dB[cols, :] as [n, h], db1[cols])."""
        X, A, b1, B, dZ = map(_f64, (X, A, b1, B, dZ))
        M, h = X.shape
        f = A.shape[1]
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        n = len(cols)
        dA_c = np.empty((h, n)); dB_r = np.empty((n, h)); db1_c = np.empty(n)
        self.lib.oracle_bwd_ffn_cols(M, h, f, act, _ptr(X), _ptr(A), _ptr(b1), _ptr(B), _ptr(dZ),
                                     n, _ptr(cols), _ptr(dA_c), _ptr(dB_r), _ptr(db1_c))
        return dA_c, dB_r, db1_c

    def linear_fwd(self, X, W, b=None):
        """Y = X W + b."""
        X, W, b = _f64(X), _f64(W), _f64(b)
        M, K = X.shape
        N = W.shape[1]
        Y = np.empty((M, N))
        self.lib.oracle_linear_fwd(M, K, N, _ptr(X), _ptr(W), _ptr(b), _ptr(Y))
        return Y

    def linear_bwd(self, X, W, dY, with_bias=True):
        """Returns (dX, dW, db) of Y = X W + b."""
        X, W, dY = _f64(X), _f64(W), _f64(dY)
        M, K = X.shape
        N = W.shape[1]
        dX = np.empty((M, K)); dW = np.empty((K, N)); db = np.empty(N) if with_bias else None
        self.lib.oracle_linear_bwd(M, K, N, _ptr(X), _ptr(W), _ptr(dY), _ptr(dX), _ptr(dW), _ptr(db))
        return dX, dW, db

    def silu(self, x: float) -> float:
        return float(self.lib.oracle_silu(float(x)))

    def silu_grad(self, x: float) -> float:
        return float(self.lib.oracle_silu_grad(float(x)))

    def swiglu_fwd(self, X, G, U, bg, bu, B, b2):
        """Returns (Hg, Hu, Y, Z) of the SwiGLU block."""
        X, G, U, bg, bu, B, b2 = map(_f64, (X, G, U, bg, bu, B, b2))
        M, h = X.shape
        f = G.shape[1]
        Hg = np.empty((M, f)); Hu = np.empty((M, f)); Y = np.empty((M, f)); Z = np.empty((M, h))
        self.lib.oracle_swiglu_fwd(M, h, f, _ptr(X), _ptr(G), _ptr(U), _ptr(bg), _ptr(bu), _ptr(B), _ptr(b2),
                                   _ptr(Hg), _ptr(Hu), _ptr(Y), _ptr(Z))
        return Hg, Hu, Y, Z

    def swiglu_bwd(self, X, G, U, B, Hg, Hu, Y, dZ):
        """Returns dict dX, dG, dU, dB, dbg, dbu, db2."""
        X, G, U, B, Hg, Hu, Y, dZ = map(_f64, (X, G, U, B, Hg, Hu, Y, dZ))
        M, h = X.shape
        f = G.shape[1]
        out = {k: np.empty(sh) for k, sh in (("dX", (M, h)), ("dG", (h, f)), ("dU", (h, f)), ("dB", (f, h)),
                                             ("dbg", (f,)), ("dbu", (f,)), ("db2", (h,)))}
        work = np.empty(3 * M * f + M * h)
        self.lib.oracle_swiglu_bwd(M, h, f, _ptr(X), _ptr(G), _ptr(U), _ptr(B), _ptr(Hg), _ptr(Hu), _ptr(Y),
                                   _ptr(dZ), _ptr(out["dX"]), _ptr(out["dG"]), _ptr(out["dU"]), _ptr(out["dB"]),
                                   _ptr(out["dbg"]), _ptr(out["dbu"]), _ptr(out["db2"]), _ptr(work))
        return out

    def swiglu_pack(self, G, U, p):
        """[rows, f] gate and up -> packed [p, rows, 2 f/p] (128-feature blocks)."""
        G = np.ascontiguousarray(G); U = np.ascontiguousarray(U)
        rows, f = G.shape
        out = np.empty((p, rows, 2 * (f // p)), dtype=G.dtype)
        self.lib.oracle_swiglu_pack(G.itemsize, rows, f, p, 0, _ptr(G), _ptr(U), _ptr(out))
        return out

    def swiglu_unpack(self, W, p):
        W = np.ascontiguousarray(W)
        _, rows, c2 = W.shape
        f = c2 // 2 * p
        G = np.empty((rows, f), dtype=W.dtype); U = np.empty((rows, f), dtype=W.dtype)
        self.lib.oracle_swiglu_pack(W.itemsize, rows, f, p, 1, _ptr(G), _ptr(U), _ptr(W))
        return G, U

    def bwd_db2(self, dZ):
        """db2 = column sums of dZ."""
        dZ = _f64(dZ)
        M, h = dZ.shape
        out = np.empty(h)
        self.lib.oracle_bwd_db2(M, h, _ptr(dZ), _ptr(out))
        return out

    def shard_columns(self, W, p):
        """[rows, cols] -> [p, rows, cols/p] (element words copied verbatim)."""
        W = np.ascontiguousarray(W)
        rows, cols = W.shape
        out = np.empty((p, rows, cols // p), dtype=W.dtype)
        self.lib.oracle_shard_columns(W.itemsize, rows, cols, p, _ptr(W), _ptr(out))
        return out

    def qkv_src_col(self, dst_col, h, n_heads) -> int:
        return int(self.lib.oracle_qkv_src_col(dst_col, h, n_heads))

    def qkv_interleave(self, W, h, n_heads, inverse=False):
        """Per-head interleave of a packed [rows, 3h] QKV weight (or its inverse)."""
        W = np.ascontiguousarray(W)
        rows, cols = W.shape
        assert cols == 3 * h
        out = np.empty_like(W)
        self.lib.oracle_qkv_interleave(W.itemsize, rows, h, n_heads, int(bool(inverse)), _ptr(W), _ptr(out))
        return out


_default = None


def get() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
