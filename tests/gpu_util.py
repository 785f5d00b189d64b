"""Shared helpers of the GPU parity tests: tolerances and oracle references.

Tolerances (per output tensor, against the fp64 oracle on the same inputs):
  bf16 path: relative Frobenius error <= 3e-3, and every element's error beyond the rounding
             of its own bf16 store within 3e-2 * max(1, RMS(ref)):
                 |got - ref| <= 3e-2 * max(1, RMS(ref)) + u(ref)
             where u(ref) is half the spacing of bf16 numbers at |ref| (2^(e-8) for
             |ref| in [2^e, 2^(e+1))) if the output is stored in bf16, else 0.
             A bf16 output of magnitude 8..16 already carries a rounding error up to
             2^-5 = 0.031 > 0.03, and heavy-tailed outputs (the SwiGLU product of two
             Gaussians) reach magnitudes far above their RMS; at RMS <= 1 and |ref| < 8 the
             bound is the literal 3e-2 plus at most the store's own rounding.
  fp32 path: relative Frobenius error <= 1e-5.
"""
from __future__ import annotations

import numpy as np

REL_F_BF16 = 3e-3
ABS_BF16 = 3e-2
REL_F_F32 = 1e-5


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    d = got - ref
    nref = np.linalg.norm(ref)
    rel_f = np.linalg.norm(d) / nref if nref > 0 else np.linalg.norm(d)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    return rel_f, max_abs, rms


def stored_as_bf16(got) -> bool:
    """True when every value is exactly a bf16 number (the low 16 bits of its fp32 form are 0)."""
    f32 = np.asarray(got, dtype=np.float32)
    return bool(np.all((f32.view(np.uint32) & np.uint32(0xFFFF)) == 0))


def bf16_half_spacing(a):
    """Half the spacing of bf16 numbers at magnitude |a| (8 significant bits): 2^(e-8) for
    |a| in [2^e, 2^(e+1)); the smallest normal spacing below 2^-126."""
    a = np.maximum(np.abs(np.asarray(a, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def assert_close(got, ref, dtype="bf16", name=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rel_f, max_abs, rms = errors(got, ref)
    if dtype == "bf16":
        assert rel_f <= REL_F_BF16, f"{name}: rel Frobenius {rel_f:.3e} > {REL_F_BF16}"
        bound = ABS_BF16 * max(1.0, rms)
        excess = np.abs(got - ref)
        if got.size and stored_as_bf16(got):
            excess = excess - bf16_half_spacing(np.maximum(np.abs(ref), np.abs(got)))
        worst = float(np.max(excess)) if excess.size else 0.0
        assert worst <= bound, (f"{name}: max abs {max_abs:.3e}, beyond the bf16 store's rounding "
                                f"{worst:.3e} > {bound:.3e} (rms {rms:.3e})")
    else:
        assert rel_f <= REL_F_F32, f"{name}: rel Frobenius {rel_f:.3e} > {REL_F_F32}"
    return rel_f, max_abs


def host_inputs_f64(buf):
    """fp64 values of the workload's unsharded inputs (exact widening)."""
    from megatron_tensor_mlp_gb300 import synth
    h = buf.host
    return {k: (None if v is None else synth.widen(v)) for k, v in h.items()}
