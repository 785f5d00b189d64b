"""The seeded input generator (CPU only)."""
import numpy as np

from megatron_tensor_mlp_gb300 import synth


def test_deterministic_and_windowed():
    a = synth.normal(3, synth.STREAM_X, (64, 40), 1.0, "bf16")
    b = synth.normal(3, synth.STREAM_X, (64, 40), 1.0, "bf16")
    assert np.array_equal(a, b)
    # a row window drawn with an offset equals the same rows of the full tensor
    w = synth.normal(3, synth.STREAM_X, (10, 40), 1.0, "bf16", offset=17 * 40)
    assert np.array_equal(w, a[17:27])
    # different streams / seeds differ
    assert not np.array_equal(a, synth.normal(3, synth.STREAM_A, (64, 40), 1.0, "bf16"))
    assert not np.array_equal(a, synth.normal(4, synth.STREAM_X, (64, 40), 1.0, "bf16"))


def test_moments():
    x = synth.widen(synth.normal(0, synth.STREAM_B, (200_000,), 0.02, "bf16"))
    assert abs(x.mean()) < 0.02 * 0.01
    assert abs(x.std() / 0.02 - 1.0) < 0.01
    y = synth.widen(synth.normal(0, synth.STREAM_X, (200_000,), 1.0, "f32"))
    assert abs(y.std() - 1.0) < 0.01
    # fourth moment of a normal is 3 sigma^4
    assert abs(np.mean(y ** 4) - 3.0) < 0.1


def test_bf16_rounding_is_nearest_even():
    f = synth.normal(5, synth.STREAM_X, (4096,), 1.0, "f32").astype(np.float32)
    b = synth.normal(5, synth.STREAM_X, (4096,), 1.0, "bf16")
    fb = synth.widen(b)
    # the bf16 value is the nearest bf16 to the fp32 draw
    u = f.view(np.uint32).astype(np.uint64)
    lo = ((u >> 16) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    hi_bits = (((u >> 16) + 1) << 16).astype(np.uint32)
    hi = hi_bits.view(np.float32).astype(np.float64)
    d_lo = np.abs(f - lo)
    d_hi = np.abs(f - hi)
    best = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    assert np.array_equal(fb[~tie], best[~tie])


def test_workloads():
    w = synth.WORKLOADS[4]
    assert (w.M, w.h, w.ffn, w.p) == (4096, 8192, 32768, 8)
    assert abs(w.fwd_flops() - 4.398e12) < 1e9
    assert synth.WORKLOADS[1].dtype == "f32" and synth.WORKLOADS[1].seed == 0
    t = synth.custom(3, 5, 16, 48, 3)
    X = t.gen("X")
    assert X.shape == (15, 16) and X.dtype == np.uint16
