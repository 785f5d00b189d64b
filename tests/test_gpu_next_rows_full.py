"""The SwiGLU block and the attention projections at the benchmark's full size (s=2048, b=4,
h=5120, p=4; ffn=20480 per SwiGLU branch, 40 heads), in the launch configuration the bench
times, against the oracle on sampled outputs (GPU).

Every GEMM here runs several waves of CTA-pair tiles, so second-wave tiles that walk K
backwards are covered too.  The oracle is evaluated on slices that determine the sampled
outputs exactly: forward outputs and input gradients are row-local (a few token rows with all
weights), weight and bias gradients are feature-local (all tokens with a few output features).
"""
import numpy as np
import pytest

import gpu_util as U

pytestmark = pytest.mark.gpu

S, B_, H, F, P, HEADS = 2048, 4, 5120, 20480, 4, 40
M = S * B_


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth, tpmlp
    return harness, synth, tpmlp


def _rows(n, seed):
    rng = np.random.default_rng(seed)
    return np.array(sorted({0, 1, M // 2, M - 1} | set(rng.integers(0, M, n).tolist())), dtype=np.int64)


def _cols(total, n, seed):
    rng = np.random.default_rng(seed)
    return np.array(sorted({0, 127, 128, total - 1} | set(rng.integers(0, total, n).tolist())), dtype=np.int64)


def test_swiglu_full_size_sampled(env, orc):
    import torch
    harness, synth, T = env
    fs = F // P
    gen = lambda sid, shp, sig: synth.normal(91, sid, shp, sig, "bf16")  # noqa: E731
    X, G, Uw, B = gen(1, (M, H), 1.0), gen(2, (H, F), 0.02), gen(9, (H, F), 0.02), gen(3, (F, H), 0.02)
    bg, bu, b2, dZ = gen(4, (F,), 0.05), gen(10, (F,), 0.05), gen(5, (H,), 0.05), gen(6, (M, H), 1.0)
    d = harness.to_torch
    W = torch.empty((P, H, 2 * fs), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_swiglu_pack(d(G), d(Uw), W, H, F, P)
    bw = torch.empty((P, 2 * fs), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_swiglu_pack(d(bg), d(bu), bw, 1, F, P)
    Bd = d(B).view(P, fs, H)
    Z = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((P, M, fs), dtype=torch.bfloat16, device="cuda")
    Hs = torch.empty((P, M, 2 * fs), dtype=torch.float32, device="cuda")
    Xd, dZd = d(X), d(dZ)
    T.tpmlp_swiglu_mlp_fwd(Xd, W, bw, Bd, d(b2), Z, Y, Hs, S, B_, H, F, P)
    dX = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((P, H, 2 * fs), dtype=torch.float32, device="cuda")
    dB = torch.empty((P, fs, H), dtype=torch.float32, device="cuda")
    dbw = torch.empty((P, 2 * fs), dtype=torch.float32, device="cuda")
    db2 = torch.empty((H,), dtype=torch.float32, device="cuda")
    dH = torch.empty((P, M, 2 * fs), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_swiglu_mlp_bwd(Xd, W, Bd, Hs, Y, dZd, dX, dW, dB, dbw, db2, dH, S, B_, H, F, P)
    T.tpmlp_device_status()
    x = synth.widen
    Xf, Gf, Uf, Bf, dZf = x(X), x(G), x(Uw), x(B), x(dZ)
    bgf, buf_, b2f = x(bg), x(bu), x(b2)

    # row-local: forward outputs and dX of sampled tokens, with all weights
    rows = _rows(8, 1)
    Hg_r, Hu_r, Y_r, Z_r = orc.swiglu_fwd(Xf[rows], Gf, Uf, bgf, buf_, Bf, b2f)
    ridx = torch.from_numpy(rows).cuda()
    U.assert_close(harness.to_host(Z[ridx]), Z_r, "bf16", "Z rows")
    U.assert_close(harness.to_host(Y.permute(1, 0, 2)[ridx].reshape(len(rows), F)), Y_r, "bf16", "Y rows")
    Hg_gpu, Hu_gpu = orc.swiglu_unpack(harness.to_host(Hs.permute(1, 0, 2)[ridx]).transpose(1, 0, 2).copy(), P)
    assert np.max(np.abs(Hg_gpu - Hg_r)) <= 1e-5 * max(1.0, np.max(np.abs(Hg_r)))
    assert np.max(np.abs(Hu_gpu - Hu_r)) <= 1e-5 * max(1.0, np.max(np.abs(Hu_r)))
    g_rows = orc.swiglu_bwd(Xf[rows], Gf, Uf, Bf, Hg_r, Hu_r, Y_r, dZf[rows])
    U.assert_close(harness.to_host(dX[ridx]), g_rows["dX"], "bf16", "dX rows")

    # feature-local: weight and bias gradients of sampled features, over all tokens
    cols = _cols(F, 8, 2)
    Hg_c, Hu_c, Y_c, _ = orc.swiglu_fwd(Xf, Gf[:, cols], Uf[:, cols], bgf[cols], buf_[cols], Bf[cols], b2f)
    g_cols = orc.swiglu_bwd(Xf, Gf[:, cols], Uf[:, cols], Bf[cols], Hg_c, Hu_c, Y_c, dZf)
    dG_gpu, dU_gpu = orc.swiglu_unpack(harness.to_host(dW), P)
    U.assert_close(dG_gpu[:, cols], g_cols["dG"], "bf16", "dG cols")
    U.assert_close(dU_gpu[:, cols], g_cols["dU"], "bf16", "dU cols")
    U.assert_close(harness.to_host(dB.reshape(F, H))[cols], g_cols["dB"], "bf16", "dB rows")
    dbg_gpu, dbu_gpu = orc.swiglu_unpack(harness.to_host(dbw).reshape(P, 1, 2 * fs), P)
    U.assert_close(dbg_gpu.reshape(-1)[cols], g_cols["dbg"], "bf16", "dbg")
    U.assert_close(dbu_gpu.reshape(-1)[cols], g_cols["dbu"], "bf16", "dbu")
    U.assert_close(harness.to_host(db2), orc.bwd_db2(dZf), "bf16", "db2")
    for t in (Z, dX, dW, dB):
        assert bool(torch.isfinite(t).all())


def test_attention_projections_full_size_sampled(env, orc):
    import torch
    harness, synth, T = env
    h3, hp = 3 * H, H // P
    gen = lambda sid, shp, sig: synth.normal(92, sid, shp, sig, "bf16")  # noqa: E731
    X, Wq, bq = gen(1, (M, H), 1.0), gen(2, (H, h3), 0.02), gen(4, (h3,), 0.05)
    dQ, ctx, Wo, bo, dZ = gen(6, (M, h3), 1.0), gen(7, (M, H), 1.0), gen(3, (H, H), 0.02), gen(5, (H,), 0.05), \
        gen(8, (M, H), 1.0)
    d = harness.to_torch
    Xd = d(X)
    # QKV: per-head interleave, column shards, column layer without activation
    Wi = torch.empty((H, h3), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_qkv_interleave(d(Wq), Wi, H, H, HEADS, P)
    bi = torch.empty((h3,), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_qkv_interleave(d(bq), bi, 1, H, HEADS, P)
    W_sh = torch.empty((P, H, h3 // P), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_shard_columns(Wi, W_sh, H, h3, P)
    QKV = torch.empty((P, M, h3 // P), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_column_fwd(Xd, W_sh, bi, QKV, None, S, B_, H, h3, P, act=T.ACT_NONE)
    dQd = d(dQ).view(M, P, h3 // P).permute(1, 0, 2).contiguous()
    dX = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    dW_sh = torch.empty((P, H, h3 // P), dtype=torch.float32, device="cuda")
    db_sh = torch.empty((P, h3 // P), dtype=torch.float32, device="cuda")
    T.tpmlp_column_bwd(Xd, W_sh, dQd, dX, dW_sh, db_sh, S, B_, H, h3, P)
    # output projection: row layer over the ranks' head blocks
    ctx_sh = d(ctx).view(M, P, hp).permute(1, 0, 2).contiguous()
    Wo_d = d(Wo)
    Z = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_row_fwd(ctx_sh, Wo_d, d(bo), Z, S, B_, H, H, P)
    dctx = torch.empty((P, M, hp), dtype=torch.bfloat16, device="cuda")
    dWo = torch.empty((P, hp, H), dtype=torch.float32, device="cuda")
    dbo = torch.empty((H,), dtype=torch.float32, device="cuda")
    T.tpmlp_row_bwd(ctx_sh, Wo_d, d(dZ), None, dctx, dWo, dbo, S, B_, H, H, P, act=T.ACT_NONE)
    T.tpmlp_device_status()
    x = synth.widen
    Xf, dQf, ctxf, Wof, dZf = x(X), x(dQ), x(ctx), x(Wo), x(dZ)
    Wif = orc.qkv_interleave(x(Wq), H, HEADS)
    bif = orc.qkv_interleave(x(bq)[None, :], H, HEADS)[0]

    rows = _rows(8, 3)
    ridx = torch.from_numpy(rows).cuda()
    U.assert_close(harness.to_host(QKV.permute(1, 0, 2)[ridx].reshape(len(rows), h3)),
                   orc.linear_fwd(Xf[rows], Wif, bif), "bf16", "QKV rows")
    dX_r, _, _ = orc.linear_bwd(Xf[rows], Wif, dQf[rows])
    U.assert_close(harness.to_host(dX[ridx]), dX_r, "bf16", "dX rows (QKV)")
    U.assert_close(harness.to_host(Z[ridx]), orc.linear_fwd(ctxf[rows], Wof, x(bo)), "bf16", "Z rows (out proj)")
    dctx_r, _, _ = orc.linear_bwd(ctxf[rows], Wof, dZf[rows])
    U.assert_close(harness.to_host(dctx.permute(1, 0, 2)[ridx].reshape(len(rows), H)), dctx_r, "bf16", "dctx rows")

    cq = _cols(h3, 8, 4)
    _, dWq_c, dbq_c = orc.linear_bwd(Xf, Wif[:, cq], dQf[:, cq])
    U.assert_close(harness.to_host(dW_sh.permute(1, 0, 2).reshape(H, h3))[:, cq], dWq_c, "bf16", "dW_qkv cols")
    U.assert_close(harness.to_host(db_sh.reshape(-1))[cq], dbq_c, "bf16", "db_qkv cols")
    co = _cols(H, 8, 5)
    _, dWo_c, dbo_c = orc.linear_bwd(ctxf, Wof[:, co], dZf[:, co])
    U.assert_close(harness.to_host(dWo.reshape(H, H))[:, co], dWo_c, "bf16", "dWo cols")
    U.assert_close(harness.to_host(dbo)[co], dbo_c, "bf16", "dbo cols")
    for t in (QKV, dX, dW_sh, Z, dctx, dWo):
        assert bool(torch.isfinite(t).all())
