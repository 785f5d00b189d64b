"""SwiGLU variant of the tensor-parallel block against the oracle (GPU).

Level 2, M027: a gated activation works on local pairs of the FFN shard, so the
column + row split needs only the final sum.  Gate and up weights are packed per
shard in 128-feature blocks (tpmlp_swiglu_pack); the forward fuses
silu(gate) * up into the column GEMM's epilogue and the backward fuses the
SwiGLU derivative into the dY GEMM's epilogue.
"""
import numpy as np
import pytest

import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth, tpmlp
    return harness, synth, tpmlp


@pytest.fixture(params=[1, 2, 5], ids=["single-cta", "cta-pair", "split-k"])
def gemm_mode(request, env):
    T = env[2]
    T.tpmlp_set_gemm_mode(request.param)
    yield request.param
    T.tpmlp_set_gemm_mode(0)


@pytest.mark.parametrize("rows,ffn,p,dt", [(3, 512, 2, 0), (5, 384, 3, 0), (2, 1024, 8, 0), (4, 256, 1, 1)])
def test_pack_bitexact(env, orc, rows, ffn, p, dt):
    import torch
    _, _, T = env
    rng = np.random.default_rng(ffn + p)
    npdt = np.uint16 if dt == T.BF16 else np.uint32
    tdt = torch.int16 if dt == T.BF16 else torch.int32
    G = rng.integers(0, np.iinfo(npdt).max, size=(rows, ffn), dtype=npdt, endpoint=True)
    Uh = rng.integers(0, np.iinfo(npdt).max, size=(rows, ffn), dtype=npdt, endpoint=True)
    ref = orc.swiglu_pack(G, Uh, p)
    g = torch.from_numpy(G.view(np.int16 if dt == T.BF16 else np.int32)).cuda()
    u = torch.from_numpy(Uh.view(np.int16 if dt == T.BF16 else np.int32)).cuda()
    W = torch.full((p, rows, 2 * ffn // p), -1, dtype=tdt, device="cuda")
    T.tpmlp_swiglu_pack(g, u, W, rows, ffn, p, dt)
    g2, u2 = torch.full_like(g, -1), torch.full_like(u, -1)
    T.tpmlp_swiglu_pack(g2, u2, W, rows, ffn, p, dt, inverse=1)
    T.tpmlp_device_status()
    assert np.array_equal(W.cpu().numpy().view(npdt), ref)
    assert np.array_equal(g2.cpu().numpy().view(npdt), G) and np.array_equal(u2.cpu().numpy().view(npdt), Uh)


SHAPES = [(25, 8, 96, 768, 3), (33, 4, 128, 256, 2), (7, 3, 256, 1024, 1), (64, 4, 320, 1536, 4)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "s{}b{}h{}f{}p{}".format(*s))
def test_swiglu_fwd_bwd(env, orc, shape, gemm_mode):
    import torch
    harness, synth, T = env
    s, b, h, f, p = shape
    M, fs = s * b, f // p
    seed = sum(shape)
    gen = lambda stream, shp, sig: synth.normal(seed, stream, shp, sig, "bf16")  # noqa: E731
    X, G, Uw, B = gen(1, (M, h), 1.0), gen(2, (h, f), 0.05), gen(9, (h, f), 0.05), gen(3, (f, h), 0.05)
    bg, bu, b2, dZ = gen(4, (f,), 0.05), gen(10, (f,), 0.05), gen(5, (h,), 0.05), gen(6, (M, h), 1.0)
    d = harness.to_torch
    W = torch.empty((p, h, 2 * fs), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_swiglu_pack(d(G), d(Uw), W, h, f, p)
    bw = torch.empty((p, 2 * fs), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_swiglu_pack(d(bg), d(bu), bw, 1, f, p)
    Bd = d(B).view(p, fs, h)
    Z = torch.full((M, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((p, M, fs), float("nan"), dtype=torch.bfloat16, device="cuda")
    H = torch.full((p, M, 2 * fs), float("nan"), dtype=torch.float32, device="cuda")
    T.tpmlp_swiglu_mlp_fwd(d(X), W, bw, Bd, d(b2), Z, Y, H, s, b, h, f, p)
    dX = torch.full((M, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW = torch.full((p, h, 2 * fs), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((p, fs, h), float("nan"), dtype=torch.float32, device="cuda")
    dbw = torch.full((p, 2 * fs), float("nan"), dtype=torch.float32, device="cuda")
    db2 = torch.full((h,), float("nan"), dtype=torch.float32, device="cuda")
    dH = torch.full((p, M, 2 * fs), float("nan"), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_swiglu_mlp_bwd(d(X), W, Bd, H, Y, d(dZ), dX, dW, dB, dbw, db2, dH, s, b, h, f, p)
    T.tpmlp_device_status()
    x = synth.widen
    Hg, Hu, Yr, Zr = orc.swiglu_fwd(x(X), x(G), x(Uw), x(bg), x(bu), x(B), x(b2))
    U.assert_close(harness.to_host(Z), Zr, "bf16", "Z")
    U.assert_close(harness.to_host(Y.permute(1, 0, 2).reshape(M, f)), Yr, "bf16", "Y")
    Hg_gpu, Hu_gpu = orc.swiglu_unpack(harness.to_host(H.permute(1, 0, 2)).transpose(1, 0, 2).copy(), p)
    # fp32 pre-activations: exact up to the fp32 accumulation
    assert np.max(np.abs(Hg_gpu - Hg)) <= 1e-5 * max(1.0, np.max(np.abs(Hg)))
    assert np.max(np.abs(Hu_gpu - Hu)) <= 1e-5 * max(1.0, np.max(np.abs(Hu)))
    g = orc.swiglu_bwd(x(X), x(G), x(Uw), x(B), Hg, Hu, Yr, x(dZ))
    U.assert_close(harness.to_host(dX), g["dX"], "bf16", "dX")
    dG, dU = orc.swiglu_unpack(harness.to_host(dW), p)
    U.assert_close(dG, g["dG"], "bf16", "dG")
    U.assert_close(dU, g["dU"], "bf16", "dU")
    U.assert_close(harness.to_host(dB.reshape(f, h)), g["dB"], "bf16", "dB")
    dbg, dbu = orc.swiglu_unpack(harness.to_host(dbw).reshape(p, 1, 2 * fs), p)
    U.assert_close(dbg.reshape(-1), g["dbg"], "bf16", "dbg")
    U.assert_close(dbu.reshape(-1), g["dbu"], "bf16", "dbu")
    U.assert_close(harness.to_host(db2), g["db2"], "bf16", "db2")


def test_swiglu_rejects_bad_shapes(env):
    import torch
    _, _, T = env
    t = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    # ffn/p = 96 is not a multiple of 128
    assert T.tpmlp_swiglu_mlp_fwd(t, t, None, t, None, o, w, None, 2, 2, 64, 192, 2, check=False) == T.ERR_DIVISIBILITY
    # fp32 is not supported on this path
    assert T.tpmlp_swiglu_mlp_fwd(t, t, None, t, None, o, w, None, 2, 2, 64, 256, 2, dt=T.F32, check=False) \
        == T.ERR_DTYPE
