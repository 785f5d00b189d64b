"""The fused block forward against its two layer calls (GPU).

tpmlp_mlp_fwd runs the column GEMM and then the row GEMM with the same tiles, tile orders and
accumulation orders as tpmlp_column_fwd followed by tpmlp_row_fwd, so the two give the same bits
(at shapes whose column GEMM runs on CTA pairs with the staged epilogue and whose row GEMM runs on
split-K CTA pairs, among others).  A CUDA graph of the block forward replayed on new inputs
recomputes everything from them, and many calls in a row stay bit-identical.
"""
import pytest

pytestmark = pytest.mark.gpu

SHAPES = [(512, 4, 1024, 4096, 4), (100, 4, 512, 2048, 2), (90, 4, 520, 2080, 2)]


def _env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T
    return torch, harness, synth, T


def _layers(T, torch, buf):
    """Z, Y, H from the two layer entry points, one after the other."""
    s, b, h, f, p = buf.dims()
    Y, H, Z = torch.empty_like(buf.Y), torch.empty_like(buf.H), torch.empty_like(buf.Z)
    T.tpmlp_column_fwd(buf.X, buf.A_sh, buf.b1_sh, Y, H, s, b, h, f, p)
    T.tpmlp_row_fwd(Y, buf.B_sh, buf.b2, Z, s, b, h, f, p)
    return Z, Y, H


@pytest.mark.parametrize("shape", SHAPES, ids=["s512-h1024-p4", "ragged-p2", "ragged-h520"])
def test_block_forward_matches_layer_calls(shape):
    torch, harness, synth, T = _env()
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.03, sigma_bias=0.02, seed=71)
    buf = harness.MLPBuffers(wl, backward=True)
    for _ in range(3):
        for t in (buf.Z, buf.Y, buf.H):
            t.fill_(float("nan"))
        buf.fwd()
        Z, Y, H = _layers(T, torch, buf)
        torch.cuda.synchronize()
        T.tpmlp_device_status()
        assert torch.equal(buf.Y, Y) and torch.equal(buf.H, H) and torch.equal(buf.Z, Z)


def test_graph_replays_recompute_from_new_inputs():
    torch, harness, synth, T = _env()
    wl = synth.custom(512, 4, 1024, 4096, 4, dtype="bf16", sigma_w=0.03, sigma_bias=0.02, seed=72)
    buf = harness.MLPBuffers(wl, backward=True)
    X_a = buf.X.clone()
    X_b = torch.randn_like(buf.X.float()).mul_(0.7).to(torch.bfloat16)
    want = {}
    for name, X in (("a", X_a), ("b", X_b)):
        buf.X.copy_(X)
        Z, _, _ = _layers(T, torch, buf)
        want[name] = Z
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream
        buf.fwd(stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        buf.fwd()
    for name in ("a", "b", "a", "b", "b", "a"):
        buf.X.copy_(X_a if name == "a" else X_b)
        buf.Z.fill_(float("nan"))
        buf.Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        T.tpmlp_device_status()
        assert torch.equal(buf.Z, want[name]), name


def test_many_calls_in_a_row_stay_identical():
    torch, harness, synth, T = _env()
    wl = synth.custom(100, 4, 512, 2048, 2, dtype="bf16", sigma_w=0.03, sigma_bias=0.02, seed=73)
    buf = harness.MLPBuffers(wl, backward=True)
    Z, Y, H = _layers(T, torch, buf)
    for _ in range(150):
        buf.fwd()
    torch.cuda.synchronize()
    T.tpmlp_device_status()
    assert torch.equal(buf.Z, Z) and torch.equal(buf.Y, Y) and torch.equal(buf.H, H)
