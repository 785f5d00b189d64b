"""Shared helpers of the GPU parity tests: tolerances and oracle references.

Tolerances (per output tensor, against the fp64 oracle on the same inputs):
  bf16 path: relative Frobenius error <= 3e-3 and max |error| <= 3e-2 * max(1, RMS(ref)).
             The max-abs bound is scaled by the reference's RMS because a bf16
             output of magnitude 8..16 already carries a rounding error up to
             2^-5 = 0.031 > 0.03; at RMS <= 1 the bound is the literal 3e-2.
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


def assert_close(got, ref, dtype="bf16", name=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rel_f, max_abs, rms = errors(got, ref)
    if dtype == "bf16":
        assert rel_f <= REL_F_BF16, f"{name}: rel Frobenius {rel_f:.3e} > {REL_F_BF16}"
        bound = ABS_BF16 * max(1.0, rms)
        assert max_abs <= bound, f"{name}: max abs {max_abs:.3e} > {bound:.3e} (rms {rms:.3e})"
    else:
        assert rel_f <= REL_F_F32, f"{name}: rel Frobenius {rel_f:.3e} > {REL_F_F32}"
    return rel_f, max_abs


def host_inputs_f64(buf):
    """fp64 values of the workload's unsharded inputs (exact widening)."""
    from megatron_tensor_mlp_gb300 import synth
    h = buf.host
    return {k: (None if v is None else synth.widen(v)) for k, v in h.items()}
