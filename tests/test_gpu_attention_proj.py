"""Attention tensor-parallel projections on the column / row entry points (GPU).

The QKV projection is column parallel by heads after the per-head interleave
("Tencent Hunyuan AI Infra interview", answer on QKV; Level 2, M028); the output
projection is row parallel with the shard sum on device (Level 2, M026/M028).
Both are checked, forward and backward, against the oracle's linear layer; the
layer backward entry points are also checked to compose tpmlp_mlp_bwd exactly.
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


def _bf16(rng_seed, stream, shape, sigma, synth):
    return synth.normal(rng_seed, stream, shape, sigma, "bf16")


@pytest.fixture(params=[0, 2, 5], ids=["auto", "cta-pair", "split-k"])
def gemm_mode(request, env):
    """Automatic tiling, CTA-pair 256x256 tiles forced even where there are fewer tiles than
    co-resident pairs (every shape here), or split-K CTA pairs on the shard-summing GEMMs."""
    T = env[2]
    T.tpmlp_set_gemm_mode(request.param)
    yield request.param
    T.tpmlp_set_gemm_mode(0)


@pytest.mark.parametrize("s,b,h,n_heads,p", [(25, 8, 256, 8, 4), (50, 3, 384, 6, 3), (16, 4, 512, 16, 8)])
def test_qkv_and_output_projection(env, orc, s, b, h, n_heads, p, gemm_mode):
    import torch
    harness, synth, T = env
    M = s * b
    seed = h + n_heads
    X = _bf16(seed, 1, (M, h), 1.0, synth)
    Wqkv = _bf16(seed, 2, (h, 3 * h), 0.05, synth)
    bqkv = _bf16(seed, 4, (3 * h,), 0.05, synth)
    dQ = _bf16(seed, 6, (M, 3 * h), 1.0, synth)      # upstream gradient, in the interleaved order
    ctx = _bf16(seed, 7, (M, h), 1.0, synth)         # attention context, head-major columns
    Wo = _bf16(seed, 3, (h, h), 0.05, synth)
    bo = _bf16(seed, 5, (h,), 0.05, synth)
    dZ = _bf16(seed, 8, (M, h), 1.0, synth)
    d = harness.to_torch
    Xd, Wd, bd = d(X), d(Wqkv), d(bqkv)

    # ---- QKV projection: interleave by heads, shard columns, column layer (no activation)
    Wi = torch.empty_like(Wd)
    T.tpmlp_qkv_interleave(Wd, Wi, h, h, n_heads, p)
    bi = torch.empty_like(bd)
    T.tpmlp_qkv_interleave(bd, bi, 1, h, n_heads, p)
    W_sh = torch.empty((p, h, 3 * h // p), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_shard_columns(Wi, W_sh, h, 3 * h, p)
    QKV = torch.full((p, M, 3 * h // p), float("nan"), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_column_fwd(Xd, W_sh, bi, QKV, None, s, b, h, 3 * h, p, act=T.ACT_NONE)
    T.tpmlp_device_status()
    x = synth.widen
    ref = orc.qkv_interleave(orc.linear_fwd(x(X), x(Wqkv), x(bqkv)), h, n_heads)
    got = harness.to_host(QKV.permute(1, 0, 2).reshape(M, 3 * h))
    U.assert_close(got, ref, "bf16", "QKV")

    # ---- QKV projection backward (column layer): dW local per rank, dX summed on device
    dQd = d(dQ).view(M, p, 3 * h // p).permute(1, 0, 2).contiguous()   # rank layout [p][M][3h/p]
    dX = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    dW_sh = torch.empty((p, h, 3 * h // p), dtype=torch.float32, device="cuda")
    db_sh = torch.empty((p, 3 * h // p), dtype=torch.float32, device="cuda")
    T.tpmlp_column_bwd(Xd, W_sh, dQd, dX, dW_sh, db_sh, s, b, h, 3 * h, p)
    T.tpmlp_device_status()
    Wi_h = orc.qkv_interleave(x(Wqkv), h, n_heads)
    rdX, rdW, rdb = orc.linear_bwd(x(X), Wi_h, x(dQ))
    U.assert_close(harness.to_host(dX), rdX, "bf16", "dX (QKV)")
    U.assert_close(harness.to_host(dW_sh.permute(1, 0, 2).reshape(h, 3 * h)), rdW, "bf16", "dW_qkv")
    U.assert_close(harness.to_host(db_sh.reshape(-1)), rdb, "bf16", "db_qkv")

    # ---- output projection: row layer over the ranks' head blocks, shard sum on device
    ctx_sh = d(ctx).view(M, p, h // p).permute(1, 0, 2).contiguous()
    Wo_d, bo_d = d(Wo), d(bo)
    Z = torch.full((M, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_row_fwd(ctx_sh, Wo_d, bo_d, Z, s, b, h, h, p)
    T.tpmlp_device_status()
    U.assert_close(harness.to_host(Z), orc.linear_fwd(x(ctx), x(Wo), x(bo)), "bf16", "Z (out proj)")

    # ---- output projection backward (row layer, no activation)
    dctx = torch.empty((p, M, h // p), dtype=torch.bfloat16, device="cuda")
    dWo = torch.empty((p, h // p, h), dtype=torch.float32, device="cuda")
    dbo = torch.empty((h,), dtype=torch.float32, device="cuda")
    T.tpmlp_row_bwd(ctx_sh, Wo_d, d(dZ), None, dctx, dWo, dbo, s, b, h, h, p, act=T.ACT_NONE)
    T.tpmlp_device_status()
    rdc, rdWo, rdbo = orc.linear_bwd(x(ctx), x(Wo), x(dZ))
    U.assert_close(harness.to_host(dctx.permute(1, 0, 2).reshape(M, h)), rdc, "bf16", "dctx")
    U.assert_close(harness.to_host(dWo.reshape(h, h)), rdWo, "bf16", "dWo")
    U.assert_close(harness.to_host(dbo), rdbo, "bf16", "dbo")


def test_layer_backwards_compose_mlp_bwd(env, orc):
    """tpmlp_mlp_bwd == tpmlp_row_bwd(GeLU') then tpmlp_column_bwd, bit for bit."""
    import torch
    harness, synth, T = env
    wl = synth.custom(40, 6, 192, 768, 3, dtype="bf16", seed=31)
    buf = harness.MLPBuffers(wl, backward=True)
    s, b, h, f, p = buf.dims()
    buf.fwd()
    buf.bwd()
    dH = torch.empty_like(buf.dH)
    dB = torch.empty_like(buf.dB_sh)
    db2 = torch.empty_like(buf.db2)
    T.tpmlp_row_bwd(buf.Y, buf.B_sh, buf.dZ, buf.H, dH, dB, db2, s, b, h, f, p, act=T.ACT_GELU_ERF)
    dX = torch.empty_like(buf.dX)
    dA = torch.empty_like(buf.dA_sh)
    db1 = torch.empty_like(buf.db1_sh)
    T.tpmlp_column_bwd(buf.X, buf.A_sh, dH, dX, dA, db1, s, b, h, f, p)
    T.tpmlp_device_status()
    for a, b_ in ((dH, buf.dH), (dB, buf.dB_sh), (db2, buf.db2), (dX, buf.dX), (dA, buf.dA_sh), (db1, buf.db1_sh)):
        assert torch.equal(a, b_)


def test_sequence_parallel_layout_is_row_blocks(env, orc):
    """Sequence parallelism (Level 2, M034: the row layer's Reduce-Scatter leaves rank r
    the sequence positions r*s/p .. (r+1)*s/p - 1 of the [s, b, h] output).  With
    tokens ordered m = s_idx * b + b_idx, rank r's sequence shard of Z is the
    contiguous row block r of Z viewed as [p][s/p * b][h]; likewise the All-Gather
    before the column layer is the identity on X.  Checked token by token."""
    harness, synth, T = env
    s, b, h, f, p = 32, 3, 128, 512, 4
    wl = synth.custom(s, b, h, f, p, dtype="bf16", seed=33)
    buf = harness.MLPBuffers(wl, backward=False)
    buf.fwd()
    T.tpmlp_device_status()
    x = U.host_inputs_f64(buf)
    _, _, Z = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    Zsp = harness.to_host(buf.Z.view(p, (s // p) * b, h))
    for r in range(p):
        rows = [s_idx * b + b_idx for s_idx in range(r * s // p, (r + 1) * s // p) for b_idx in range(b)]
        U.assert_close(Zsp[r], Z[rows], "bf16", f"sequence shard {r}")
