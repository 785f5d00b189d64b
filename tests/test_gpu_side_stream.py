"""The fused backward with a side stream of the caller's (GPU).

With a stream and two events registered (tpmlp_set_side_stream), tpmlp_mlp_bwd at the s=512 b=4
h=1024 ffn=4096 p=4 workload (every GEMM one or two waves of tiles; also a ragged shape near it)
runs its two pairs of independent GEMMs side by side, dH beside dB and dA beside dX, each on a
share of the SMs; with nothing registered everything runs in line on one stream.  Each tile keeps its accumulation order
on the smaller grids, so dH, dB, dA and the column sums db1, db2 have the same bits both ways.
dX runs on CTA pairs over its whole K loop in its share, rather than on split-K pairs that add
two fp32 halves, so a few of its bf16 values round the other way: it is checked against the
in-line result to one bf16 step, and against the unsharded sum.  At the bench's sizes (GEMMs of
many waves) the side stream instead takes the column sums beside the weight-gradient GEMMs'
split-K last waves, in the GeLU and the SwiGLU block: there every output keeps its bits.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(512, 4, 1024, 4096, 4), (250, 4, 1032, 4128, 4)], ids=["s512-h1024", "ragged"])
def test_side_stream_sums_are_bit_identical(shape):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.02, sigma_bias=0.01, seed=66)
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
    for name, a, b in zip(("db1", "db2", "dA", "dB", "dH"), ref[:2] + ref[3:], outs[:2] + outs[3:]):
        assert torch.equal(a, b), name
    # dX: the same sums in another fp32 order, each rounded to bf16 once: one bf16 step apart,
    # or, where the sum of 4096 products cancels to a small value, within the fp32 order's
    # error, far below the values' own scale
    dx_ref, dx = ref[2].float(), outs[2].float()
    rms = float(torch.sqrt((dx_ref * dx_ref).mean()))
    step = torch.maximum(dx_ref.abs(), dx.abs()) * 2.0 ** -7 + 1e-3 * rms
    assert bool(((dx - dx_ref).abs() <= step).all())
    assert float((dx != dx_ref).float().mean()) < 0.05
    want_dx = torch.einsum("imf,ihf->mh", buf.dH.float(), buf.A_sh.float())
    assert float(torch.linalg.norm(dx - want_dx) / torch.linalg.norm(want_dx)) < 5e-3
    db2 = harness.to_host(buf.db2)
    want = synth.widen(buf.host["dZ"]).sum(axis=0)
    assert np.linalg.norm(db2 - want) / np.linalg.norm(want) < 1e-5


@pytest.mark.parametrize("shape", [(2048, 4, 5120, 20480, 4), (2050, 4, 5120, 20480, 4)], ids=["bench", "ragged-M"])
def test_sums_beside_last_waves_are_bit_identical(shape):
    """At the fwd+bwd bench workload (s=2048 b=4 h=5120 ffn=20480 p=4) every GEMM spans many waves, so
    the backward runs its GEMMs in line; dB_i and dA_i end on a split-K last wave of 4 tiles on 16
    SMs, and with a side stream registered the column sums run beside those last waves (db2 beside
    dB's, db1 beside dA's).  Every output keeps its bits, dX included; the outputs are poisoned
    first and checked after a single call, so sums that read dH before it is complete would show.
    The second shape has 8 tokens past a 256-row block (a ragged K for dB and dA, ragged rows for
    the other GEMMs) and the same last waves."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.02, sigma_bias=0.01, seed=67)
    buf = harness.MLPBuffers(wl, backward=True)
    buf.fwd()
    buf.bwd()
    torch.cuda.synchronize()
    T.tpmlp_device_status()
    names = ("db1", "db2", "dX", "dA", "dB", "dH")
    outs = (buf.db1_sh, buf.db2, buf.dX, buf.dA_sh, buf.dB_sh, buf.dH)
    ref = [t.clone() for t in outs]
    side, fork, join = torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()
    T.tpmlp_set_side_stream(side, fork, join)
    try:
        for rep in range(3):
            for t in outs:
                t.fill_(float("nan"))
            buf.bwd()
            torch.cuda.synchronize()
            T.tpmlp_device_status()
            for name, a, b in zip(names, ref, outs):
                assert torch.equal(a, b), f"{name} (call {rep})"
    finally:
        T.tpmlp_set_side_stream(None, None, None)


def test_swiglu_sums_beside_last_waves_are_bit_identical():
    """The SwiGLU block backward at the bench's sizes (s=2048 b=4 h=5120, ffn=20480 per branch, p=4):
    dB_i and the packed dW_i end on split-K last waves (4 and 8 tiles), so with a side stream
    registered db2 runs beside dB's and the packed bias gradient beside dW's.  Every output keeps
    its bits against the in-line run, after single calls on poisoned buffers."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import tpmlp as T

    s, b, h, f, p = 2048, 4, 5120, 20480, 4
    M, fs, bf = s * b, f // p, torch.bfloat16
    g = torch.Generator(device="cuda").manual_seed(68)
    rnd = lambda shape, sig: (torch.randn(shape, generator=g, device="cuda") * sig).to(bf)  # noqa: E731
    X, dZ = rnd((M, h), 1.0), rnd((M, h), 1.0)
    W, bw, B = rnd((p, h, 2 * fs), 0.02), rnd((p, 2 * fs), 0.01), rnd((p, fs, h), 0.02)
    Z, Y = torch.empty((M, h), dtype=bf, device="cuda"), torch.empty((p, M, fs), dtype=bf, device="cuda")
    H = torch.empty((p, M, 2 * fs), dtype=torch.float32, device="cuda")
    T.tpmlp_swiglu_mlp_fwd(X, W, bw, B, None, Z, Y, H, s, b, h, f, p)
    dX, dH = torch.empty((M, h), dtype=bf, device="cuda"), torch.empty((p, M, 2 * fs), dtype=bf, device="cuda")
    dW = torch.empty((p, h, 2 * fs), dtype=torch.float32, device="cuda")
    dB = torch.empty((p, fs, h), dtype=torch.float32, device="cuda")
    dbw, db2 = torch.empty((p, 2 * fs), dtype=torch.float32, device="cuda"), torch.empty(h, dtype=torch.float32,
                                                                                            device="cuda")
    outs = (dX, dW, dB, dbw, db2, dH)
    names = ("dX", "dW", "dB", "dbw", "db2", "dH")

    def bwd():
        T.tpmlp_swiglu_mlp_bwd(X, W, B, H, Y, dZ, dX, dW, dB, dbw, db2, dH, s, b, h, f, p)

    bwd()
    torch.cuda.synchronize()
    T.tpmlp_device_status()
    ref = [t.clone() for t in outs]
    side, fork, join = torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()
    T.tpmlp_set_side_stream(side, fork, join)
    try:
        for rep in range(2):
            for t in outs:
                t.fill_(float("nan"))
            bwd()
            torch.cuda.synchronize()
            T.tpmlp_device_status()
            for name, a, c in zip(names, ref, outs):
                assert torch.equal(a, c), f"{name} (call {rep})"
    finally:
        T.tpmlp_set_side_stream(None, None, None)
