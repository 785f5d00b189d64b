"""Column sums of the fused backward on a side stream of the caller's (GPU).

With a stream and two events registered (tpmlp_set_side_stream), tpmlp_mlp_bwd runs db1 and db2
on that stream beside the first of the dA and dX GEMMs whose grid leaves enough SMs idle for all
the sums' CTAs; with nothing registered they run in line.  Both give the same bits, and every
other output is unchanged.  The shape is the s=512 b=4 h=1024 ffn=4096 p=4 workload: its dA GEMM
runs 128 single-CTA tiles on the 152 SMs, and the sums need 20 CTAs (16 strips of db1, 4 of db2),
so they go beside dA.
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

    wl = synth.custom(512, 4, 1024, 4096, 4, dtype="bf16", sigma_w=0.02, sigma_bias=0.01, seed=66)
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
