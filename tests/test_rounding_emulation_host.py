"""The rounding-point comparison of test_gpu_rounding.py can tell protocols apart (CPU).

The GPU test allows at most MAX_FLIP_FRACTION of a bf16 output's elements to sit one unit from
the emulation of reading r7.  Here the emulation is compared with the same emulation under the
two plausible wrong protocols, on the GPU test's own inputs: GeLU taken of the saved bf16 H
instead of the fp32 one, and GeLU' taken of the fp32 H instead of the saved one.  Each moves
many times that fraction of Y or dH, so neither could pass the GPU test.
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
