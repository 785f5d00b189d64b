"""The rounding-point comparison of test_gpu_rounding.py can tell protocols apart (CPU).

The GPU test allows at most MAX_FLIP_FRACTION of a bf16 output's elements to sit one unit from
the emulation of reading r7.  Here the emulation is compared with the same emulation under the
plausible wrong protocols, on the GPU tests' own inputs: GeLU taken of the saved bf16 H instead
of the fp32 one, GeLU' taken of the fp32 H instead of the saved one, and (SwiGLU) the gate and up
pre-activations saved in bf16 instead of fp32.  Each moves many times that fraction of Y, dH or
(dg, du), so none could pass the GPU test.
"""
import numpy as np

import test_gpu_rounding as R
from megatron_tensor_mlp_gb300 import synth


def _inputs():
    wl = synth.custom(64, 4, 512, 2048, 4, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=96)
    return [synth.widen(wl.gen(k)) for k in ("X", "A", "b1", "B", "b2", "dZ")]


def test_wrong_protocols_move_many_elements():
    args = _inputs()
    ok = R._emulate(*args)
    gelu_saved = R._emulate(*args, gelu_of_saved_h=True)
    grad_fp32 = R._emulate(*args, grad_of_fp32_h=True)
    frac_y = float(np.mean(gelu_saved["Y"] != ok["Y"]))
    frac_dh = float(np.mean(grad_fp32["dH"] != ok["dH"]))
    assert frac_y > 5 * R.MAX_FLIP_FRACTION, frac_y
    assert frac_dh > 5 * R.MAX_FLIP_FRACTION, frac_dh


def test_emulation_meets_the_oracle_tolerance():
    """The emulated pipeline itself is within the bf16 tolerance of the fp64 oracle."""
    import gpu_util as U
    import oracle
    orc = oracle.get()
    X, A, b1, B, b2, dZ = _inputs()
    emu = R._emulate(X, A, b1, B, b2, dZ)
    H, Y, Z = orc.mlp_fwd(X, A, b1, B, b2)
    g = orc.mlp_bwd(X, A, B, H, Y, dZ)
    for k, ref in (("Z", Z), ("Y", Y), ("H", H), ("dX", g["dX"]), ("dA", g["dA"]), ("dB", g["dB"]),
                   ("db1", g["db1"]), ("db2", g["db2"])):
        U.assert_close(emu[k], ref, "bf16", k)


def test_swiglu_bf16_saves_move_many_elements():
    gen = lambda stream, shp, sig: synth.widen(synth.normal(97, stream, shp, sig, "bf16"))  # noqa: E731
    M, h, f = 256, 512, 2048
    X, G, Uw, B = gen(1, (M, h), 1.0), gen(2, (h, f), 0.05), gen(9, (h, f), 0.05), gen(3, (f, h), 0.05)
    bg, bu, b2, dZ = gen(4, (f,), 0.05), gen(10, (f,), 0.05), gen(5, (h,), 0.05), gen(6, (M, h), 1.0)
    ok = R._emulate_swiglu(X, G, Uw, bg, bu, B, b2, dZ)
    bad = R._emulate_swiglu(X, G, Uw, bg, bu, B, b2, dZ, bf16_saves=True)
    frac = float(np.mean(np.concatenate([(bad[k] != ok[k]).ravel() for k in ("dHg", "dHu")])))
    assert frac > 5 * R.MAX_FLIP_FRACTION, frac
