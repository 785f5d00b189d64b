"""Thin ctypes binding of the tpmlp C-ABI (``include/tpmlp.h``).

Argument marshalling only: every function has the C entry point's name and
arguments; torch tensors are passed as their device pointers, ``stream``
defaults to torch's current CUDA stream.  Every step of the computation runs
in the CUDA kernels of ``libtpmlp.so``; there is no other code path, and
importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("TPMLP_LIB") or os.path.join(_HERE, "libtpmlp.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "tpmlp.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")

lib = ctypes.CDLL(LIB_PATH)

BF16, F32 = 0, 1
ACT_NONE, ACT_GELU_ERF = 0, 1

STATUS = {0: "TPMLP_OK", 1: "TPMLP_ERR_NULL", 2: "TPMLP_ERR_SHAPE", 3: "TPMLP_ERR_DIVISIBILITY",
          4: "TPMLP_ERR_DTYPE", 5: "TPMLP_ERR_ALIGNMENT", 6: "TPMLP_ERR_ALIAS", 7: "TPMLP_ERR_ARCH",
          8: "TPMLP_ERR_CUDA", 9: "TPMLP_ERR_TIMEOUT", 10: "TPMLP_ERR_DEVICE"}
OK, ERR_NULL, ERR_SHAPE, ERR_DIVISIBILITY, ERR_DTYPE, ERR_ALIGNMENT, ERR_ALIAS, ERR_ARCH, ERR_CUDA, \
    ERR_TIMEOUT, ERR_DEVICE = range(11)

_vp, _i64, _i32, _u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
_SIGS = {
    "tpmlp_column_fwd": [_vp] * 5 + [_i64] * 4 + [_i32, _i32, _i32, _vp],
    "tpmlp_row_fwd": [_vp] * 4 + [_i64] * 4 + [_i32, _i32, _vp],
    "tpmlp_mlp_fwd": [_vp] * 8 + [_i64] * 4 + [_i32, _i32, _vp],
    "tpmlp_mlp_bwd": [_vp] * 12 + [_i64] * 4 + [_i32, _i32, _i32, _vp],
    "tpmlp_mlp_fwd_noalloc": [_vp] * 6 + [_i64] * 4 + [_i32, _i32, _vp],
    "tpmlp_mlp_fwd_partial": [_vp] * 7 + [_i64] * 4 + [_i32, _i32, _vp],
    "tpmlp_mlp_bwd_partial": [_vp] * 12 + [_i64] * 4 + [_i32, _i32, _i32, _vp],
    "tpmlp_sum_finish": [_vp, _vp, _vp, _i64, _i64, _i32, _vp],
    "tpmlp_swiglu_mlp_fwd": [_vp] * 8 + [_i64] * 4 + [_i32, _i32, _vp],
    "tpmlp_swiglu_mlp_bwd": [_vp] * 12 + [_i64] * 4 + [_i32, _i32, _i32, _vp],
    "tpmlp_swiglu_pack": [_vp] * 3 + [_i64, _i64, _i32, _i32, _i32, _vp],
    "tpmlp_row_bwd": [_vp] * 7 + [_i64] * 4 + [_i32, _i32, _i32, _i32, _vp],
    "tpmlp_column_bwd": [_vp] * 6 + [_i64] * 4 + [_i32, _i32, _i32, _vp],
    "tpmlp_shard_columns": [_vp, _vp, _i64, _i64, _i32, _i32, _vp],
    "tpmlp_unshard_columns": [_vp, _vp, _i64, _i64, _i32, _i32, _vp],
    "tpmlp_qkv_interleave": [_vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32, _vp],
    "tpmlp_device_status": [_vp],
    "tpmlp_debug_wait_timeout": [_u32, _vp],
    "tpmlp_set_gemm_mode": [_i32],
    "tpmlp_set_side_stream": [_vp, _vp, _vp],
    "tpmlp_set_gemm_raster": [_i32],
    "tpmlp_set_k_chunk": [_i32],

}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.tpmlp_qkv_src_col.argtypes = [_i64, _i64, _i64]
lib.tpmlp_qkv_src_col.restype = _i64
lib.tpmlp_status_string.argtypes = [ctypes.c_int]
lib.tpmlp_status_string.restype = ctypes.c_char_p
lib.tpmlp_last_error.argtypes = []
lib.tpmlp_last_error.restype = ctypes.c_char_p
lib.tpmlp_get_gemm_raster.argtypes = []
lib.tpmlp_get_gemm_raster.restype = ctypes.c_int
lib.tpmlp_get_k_chunk.argtypes = []
lib.tpmlp_get_k_chunk.restype = ctypes.c_int
lib.tpmlp_get_gemm_mode.argtypes = []
lib.tpmlp_get_gemm_mode.restype = ctypes.c_int
lib.tpmlp_version.argtypes = []
lib.tpmlp_version.restype = ctypes.c_int
lib.tpmlp_launch_count.argtypes = []
lib.tpmlp_launch_count.restype = ctypes.c_uint64


class TpmlpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions declared in include/tpmlp.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"\b(tpmlp_[a-z0-9_]+)\s*\(", txt)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def last_error() -> str:
    return lib.tpmlp_last_error().decode()


def _done(st: int, check: bool):
    if check and st != OK:
        raise TpmlpError(st, last_error())
    return st


def tpmlp_column_fwd(X, A_sh, b1_sh, Y_sh, H_sh, s, b, h, ffn, p, dt=BF16, act=ACT_GELU_ERF, stream=None,
                     check=True):
    st = lib.tpmlp_column_fwd(_ptr(X), _ptr(A_sh), _ptr(b1_sh), _ptr(Y_sh), _ptr(H_sh), s, b, h, ffn, p, dt, act,
                              _stream(stream))
    return _done(st, check)


def tpmlp_row_fwd(Y_sh, B_sh, b2, Z, s, b, h, ffn, p, dt=BF16, stream=None, check=True):
    st = lib.tpmlp_row_fwd(_ptr(Y_sh), _ptr(B_sh), _ptr(b2), _ptr(Z), s, b, h, ffn, p, dt, _stream(stream))
    return _done(st, check)


def tpmlp_mlp_fwd(X, A_sh, b1_sh, B_sh, b2, Z, Y_ws, H_sh, s, b, h, ffn, p, dt=BF16, stream=None, check=True):
    st = lib.tpmlp_mlp_fwd(_ptr(X), _ptr(A_sh), _ptr(b1_sh), _ptr(B_sh), _ptr(b2), _ptr(Z), _ptr(Y_ws), _ptr(H_sh),
                           s, b, h, ffn, p, dt, _stream(stream))
    return _done(st, check)


def tpmlp_mlp_bwd(X, A_sh, B_sh, H_sh, Y_sh, dZ, dX, dA_sh, dB_sh, db1_sh, db2, dH_ws, s, b, h, ffn, p, dt=BF16,
                  grad_dt=F32, stream=None, check=True):
    st = lib.tpmlp_mlp_bwd(_ptr(X), _ptr(A_sh), _ptr(B_sh), _ptr(H_sh), _ptr(Y_sh), _ptr(dZ), _ptr(dX), _ptr(dA_sh),
                           _ptr(dB_sh), _ptr(db1_sh), _ptr(db2), _ptr(dH_ws), s, b, h, ffn, p, dt, grad_dt,
                           _stream(stream))
    return _done(st, check)


def tpmlp_mlp_fwd_partial(X, A_sh, b1_sh, B_sh, Z_part, Y_ws, H_sh, s, b, h, ffn, p, dt=BF16, stream=None,
                          check=True):
    """One rank's part of a block whose shards are spread over GPUs: fp32 Z_part, no b2."""
    st = lib.tpmlp_mlp_fwd_partial(_ptr(X), _ptr(A_sh), _ptr(b1_sh), _ptr(B_sh), _ptr(Z_part), _ptr(Y_ws),
                                   _ptr(H_sh), s, b, h, ffn, p, dt, _stream(stream))
    return _done(st, check)


def tpmlp_mlp_bwd_partial(X, A_sh, B_sh, H_sh, Y_sh, dZ, dX_part, dA_sh, dB_sh, db1_sh, db2, dH_ws, s, b, h, ffn, p,
                          dt=BF16, grad_dt=F32, stream=None, check=True):
    """One rank's backward: local weight and bias gradients, fp32 dX_part for the All-Reduce."""
    st = lib.tpmlp_mlp_bwd_partial(_ptr(X), _ptr(A_sh), _ptr(B_sh), _ptr(H_sh), _ptr(Y_sh), _ptr(dZ),
                                   _ptr(dX_part), _ptr(dA_sh), _ptr(dB_sh), _ptr(db1_sh), _ptr(db2), _ptr(dH_ws),
                                   s, b, h, ffn, p, dt, grad_dt, _stream(stream))
    return _done(st, check)


def tpmlp_sum_finish(S, bias, out, rows, cols, dt=BF16, stream=None, check=True):
    """out = round(S + bias) after the All-Reduce of fp32 partials."""
    return _done(lib.tpmlp_sum_finish(_ptr(S), _ptr(bias), _ptr(out), rows, cols, dt, _stream(stream)), check)


def tpmlp_swiglu_mlp_fwd(X, W_sh, bw_sh, B_sh, b2, Z, Y_ws, H_ws, s, b, h, ffn, p, dt=BF16, stream=None,
                         check=True):
    st = lib.tpmlp_swiglu_mlp_fwd(_ptr(X), _ptr(W_sh), _ptr(bw_sh), _ptr(B_sh), _ptr(b2), _ptr(Z), _ptr(Y_ws),
                                  _ptr(H_ws), s, b, h, ffn, p, dt, _stream(stream))
    return _done(st, check)


def tpmlp_swiglu_mlp_bwd(X, W_sh, B_sh, H_ws, Y_ws, dZ, dX, dW_sh, dB_sh, dbw_sh, db2, dH_ws, s, b, h, ffn, p,
                         dt=BF16, grad_dt=F32, stream=None, check=True):
    st = lib.tpmlp_swiglu_mlp_bwd(_ptr(X), _ptr(W_sh), _ptr(B_sh), _ptr(H_ws), _ptr(Y_ws), _ptr(dZ), _ptr(dX),
                                  _ptr(dW_sh), _ptr(dB_sh), _ptr(dbw_sh), _ptr(db2), _ptr(dH_ws), s, b, h, ffn, p, dt,
                                  grad_dt, _stream(stream))
    return _done(st, check)


def tpmlp_swiglu_pack(G, U, W_sh, rows, ffn, p, dt=BF16, inverse=0, stream=None, check=True):
    st = lib.tpmlp_swiglu_pack(_ptr(G), _ptr(U), _ptr(W_sh), rows, ffn, p, dt, int(inverse), _stream(stream))
    return _done(st, check)


def tpmlp_row_bwd(Y_sh, B_sh, dZ, H_sh, dY_sh, dB_sh, db2, s, b, h, ffn, p, dt=BF16, grad_dt=F32, act=ACT_NONE,
                  stream=None, check=True):
    st = lib.tpmlp_row_bwd(_ptr(Y_sh), _ptr(B_sh), _ptr(dZ), _ptr(H_sh), _ptr(dY_sh), _ptr(dB_sh), _ptr(db2), s, b, h,
                           ffn, p, dt, grad_dt, act, _stream(stream))
    return _done(st, check)


def tpmlp_column_bwd(X, A_sh, dY_sh, dX, dA_sh, db1_sh, s, b, h, ffn, p, dt=BF16, grad_dt=F32, stream=None,
                     check=True):
    st = lib.tpmlp_column_bwd(_ptr(X), _ptr(A_sh), _ptr(dY_sh), _ptr(dX), _ptr(dA_sh), _ptr(db1_sh), s, b, h, ffn,
                              p, dt, grad_dt, _stream(stream))
    return _done(st, check)


def tpmlp_mlp_fwd_noalloc(X, A_sh, b1_sh, B_sh, b2, Z, s, b, h, ffn, p, dt=BF16, stream=None, check=True):
    """The block forward with Y kept in the library's fixed array (no caller workspace)."""
    st = lib.tpmlp_mlp_fwd_noalloc(_ptr(X), _ptr(A_sh), _ptr(b1_sh), _ptr(B_sh), _ptr(b2), _ptr(Z), s, b, h, ffn, p,
                                   dt, _stream(stream))
    return _done(st, check)


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def tpmlp_shard_columns(W, W_sh, rows, cols, p, dt=BF16, stream=None, check=True):
    return _done(lib.tpmlp_shard_columns(_ptr(W), _ptr(W_sh), rows, cols, p, dt, _stream(stream)), check)


def tpmlp_unshard_columns(W_sh, W, rows, cols, p, dt=BF16, stream=None, check=True):
    return _done(lib.tpmlp_unshard_columns(_ptr(W_sh), _ptr(W), rows, cols, p, dt, _stream(stream)), check)


def tpmlp_qkv_interleave(W_qkv, W_out, rows, h, n_heads, p, dt=BF16, inverse=0, stream=None, check=True):
    st = lib.tpmlp_qkv_interleave(_ptr(W_qkv), _ptr(W_out), rows, h, n_heads, p, dt, int(inverse), _stream(stream))
    return _done(st, check)


def tpmlp_qkv_src_col(dst_col, h, n_heads) -> int:
    return int(lib.tpmlp_qkv_src_col(dst_col, h, n_heads))


def tpmlp_device_status(stream=None, check=True):
    return _done(lib.tpmlp_device_status(_stream(stream)), check)


def tpmlp_debug_wait_timeout(timeout_us, stream=None, check=True):
    return _done(lib.tpmlp_debug_wait_timeout(timeout_us, _stream(stream)), check)


# tpmlp_set_gemm_mode values
GEMM_AUTO, GEMM_SINGLE, GEMM_PAIR, GEMM_PAIR_DIRECT, GEMM_PAIR_STAGED = 0, 1, 2, 3, 4


def tpmlp_set_side_stream(side_stream, fork_event, join_event, check=True):
    """Register (or, with three Nones, clear) a side stream and two events of the caller's for the
    fused backwards: independent GEMMs side by side at small shapes, else the column sums beside a
    weight-gradient GEMM's short last wave or a GEMM that leaves SMs idle.  Torch objects or raw
    handles; the caller keeps them alive."""
    def handle(x):
        if x is None or isinstance(x, int):
            return x
        if hasattr(x, "cuda_stream"):
            return x.cuda_stream
        if not x.cuda_event:  # torch creates an event's CUDA object at its first record
            x.record(side_stream if hasattr(side_stream, "cuda_stream") else None)
        return x.cuda_event
    return _done(lib.tpmlp_set_side_stream(handle(side_stream), handle(fork_event), handle(join_event)), check)


def tpmlp_set_gemm_mode(mode, check=True):
    return _done(lib.tpmlp_set_gemm_mode(mode), check)


def tpmlp_get_gemm_mode() -> int:
    return int(lib.tpmlp_get_gemm_mode())


def tpmlp_set_gemm_raster(group_m, check=True):
    return _done(lib.tpmlp_set_gemm_raster(group_m), check)


def tpmlp_get_gemm_raster() -> int:
    return int(lib.tpmlp_get_gemm_raster())


def tpmlp_set_k_chunk(k_blocks, check=True):
    return _done(lib.tpmlp_set_k_chunk(k_blocks), check)


def tpmlp_get_k_chunk() -> int:
    return int(lib.tpmlp_get_k_chunk())


def tpmlp_status_string(st: int) -> str:
    return lib.tpmlp_status_string(st).decode()


def tpmlp_last_error() -> str:
    return last_error()


def tpmlp_version() -> int:
    return int(lib.tpmlp_version())


def tpmlp_launch_count() -> int:
    """Kernels this library has enqueued in this process so far (host-side count)."""
    return int(lib.tpmlp_launch_count())
