"""Column sums of the fused backward on a side stream of the caller's (GPU).

With a stream and two events registered (tpmlp_set_side_stream), tpmlp_mlp_bwd runs db1 and db2
beside the dX GEMM where its last wave leaves CTA pairs idle; with nothing registered they run in
line.  Both give the same bits, and every other output is unchanged.  The shape (2048 tokens,
h = 5120, ffn = 20480, p = 4) gives dX 160 CTA-pair tiles, a last wave of 8 of 76 pairs, and
2.4e-4 bytes of sums per dX flop, so the side stream is taken.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_side_stream_sums_are_bit_identical():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    wl = synth.custom(512, 4, 5120, 20480, 4, dtype="bf16", sigma_w=0.02, sigma_bias=0.0, seed=66)
    buf = harness.MLPBuffers(wl, backward=True)
    buf.fwd()
    buf.bwd()
    T.tpmlp_device_status()
    outs = (buf.db1_sh, buf.db2, buf.dX, buf.dA_sh, buf.dB_sh, buf.dH)
    ref = [t.clone() for t in outs]
    side, fork, join = torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()
    T.tpmlp_set_side_stream(side, fork, join)
    try:
        for t in outs:
            t.fill_(float("nan"))
        for _ in range(3):
            buf.bwd()
        torch.cuda.synchronize()
        T.tpmlp_device_status()
    finally:
        T.tpmlp_set_side_stream(None, None, None)
    for name, a, b in zip(("db1", "db2", "dX", "dA", "dB", "dH"), ref, outs):
        assert torch.equal(a, b), name
    db2 = harness.to_host(buf.db2)
    want = synth.widen(buf.host["dZ"]).sum(axis=0)
    assert np.linalg.norm(db2 - want) / np.linalg.norm(want) < 1e-5
