"""The five workloads at full size, in the launch configuration the benchmark
times (a side stream registered for the fused backward, as the benchmark does; the
s=512 workload with its backward too, which the benchmark also times), against the
oracle on sampled outputs computed one by one (GPU)."""
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


def _rows(M, n_random, seed):
    rng = np.random.default_rng(seed)
    r = {0, 1, 127, 128, M // 2, M - 1} | set(rng.integers(0, M, n_random).tolist())
    return np.array(sorted(x for x in r if 0 <= x < M), dtype=np.int64)


def _cols(f, p, n_random, seed):
    fs = f // p
    rng = np.random.default_rng(seed + 1)
    c = {0, fs - 1, fs, f - 1, 255, 256} | set(rng.integers(0, f, n_random).tolist())
    return np.array(sorted(x for x in c if 0 <= x < f), dtype=np.int64)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_workload_sampled(env, orc, cfg):
    import torch
    harness, synth, T = env
    wl = synth.WORKLOADS[cfg]
    backward = wl.backward or cfg == 2
    buf = harness.MLPBuffers(wl, backward=backward)
    for t in (buf.Z, buf.Y, buf.H):
        if t is not None:
            t.fill_(float("nan"))
    side = (torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event())
    T.tpmlp_set_side_stream(*side)
    try:
        buf.fwd()
        if backward:
            buf.bwd()
        torch.cuda.synchronize()
    finally:
        T.tpmlp_set_side_stream(None, None, None)
    T.tpmlp_device_status()
    M, h, f, p = wl.M, wl.h, wl.ffn, wl.p
    rows = _rows(M, 10, cfg)
    widen = synth.widen
    X = widen(buf.host["X"])
    A = widen(buf.host["A"])
    B = widen(buf.host["B"])
    b1 = None if buf.host["b1"] is None else widen(buf.host["b1"])
    b2 = None if buf.host["b2"] is None else widen(buf.host["b2"])
    Hr, Yr, Zr = orc.mlp_fwd(X[rows], A, b1, B, b2)
    ridx = torch.from_numpy(rows).cuda()
    U.assert_close(harness.to_host(buf.Z[ridx]), Zr, "bf16", f"Z rows (cfg {cfg})")
    U.assert_close(harness.to_host(buf.Y_full()[ridx]), Yr, "bf16", f"Y rows (cfg {cfg})")
    if buf.H is not None:
        U.assert_close(harness.to_host(buf.H_full()[ridx]), Hr, "bf16", f"H rows (cfg {cfg})")
    # a property at full size: every output finite
    assert bool(torch.isfinite(buf.Z).all())
    if not backward:
        return
    dZ = widen(buf.host["dZ"])
    cols = _cols(f, p, 6, cfg)
    dAc, dBr, db1c = orc.bwd_ffn_cols(X, A, b1, B, dZ, cols)
    cidx = torch.from_numpy(cols).cuda()
    U.assert_close(harness.to_host(buf.dA_full()[:, cidx]), dAc, "bf16", "dA cols")
    U.assert_close(harness.to_host(buf.dB_full()[cidx]), dBr, "bf16", "dB rows")
    U.assert_close(harness.to_host(buf.db1_sh.reshape(-1)[cidx]), db1c, "bf16", "db1")
    U.assert_close(harness.to_host(buf.db2), orc.bwd_db2(dZ), "bf16", "db2")
    xr = rows[:: max(1, len(rows) // 4)][:4]
    dXr = orc.bwd_dX_rows(X, A, b1, B, dZ, xr)
    U.assert_close(harness.to_host(buf.dX[torch.from_numpy(xr).cuda()]), dXr, "bf16", "dX rows")
    for t in (buf.dX, buf.dA_sh, buf.dB_sh):
        assert bool(torch.isfinite(t).all())


def test_offsets_past_2_31_elements_sampled(env, orc):
    """s = 2^17, b = 4 (M = 2^19 tokens), h = 128, ffn = 8192, p = 4: Y, H and dH hold 2^32
    elements each (8 GB), so element offsets past the first shards exceed 2^31 and every
    32-bit overflow in index or address arithmetic would show.  Sampled rows and columns, the
    last rows of the last shard included.  (K of the weight-gradient GEMMs is 2^19 tokens:
    the tensor cores' fp32 accumulation error grows about 1.9e-8 per 16-deep step, 6e-4 here;
    at 2^21 tokens it alone reaches 2.5e-3 of the 3e-3 bound.)"""
    import torch
    harness, synth, T = env
    wl = synth.custom(1 << 17, 4, 128, 8192, 4, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=2019)
    buf = harness.MLPBuffers(wl, backward=True)
    buf.fwd()
    buf.bwd()
    T.tpmlp_device_status()
    M, h, f, p = wl.M, wl.h, wl.ffn, wl.p
    rng = np.random.default_rng(5)
    rows = np.array(sorted({0, M // 2, M - 2, M - 1} | set(rng.integers(0, M, 8).tolist())), dtype=np.int64)
    widen = synth.widen
    X, A, B = widen(buf.host["X"]), widen(buf.host["A"]), widen(buf.host["B"])
    b1, b2, dZ = widen(buf.host["b1"]), widen(buf.host["b2"]), widen(buf.host["dZ"])
    Hr, Yr, Zr = orc.mlp_fwd(X[rows], A, b1, B, b2)
    ridx = torch.from_numpy(rows).cuda()
    U.assert_close(harness.to_host(buf.Z[ridx]), Zr, "bf16", "Z rows")
    U.assert_close(harness.to_host(buf.Y_full()[ridx]), Yr, "bf16", "Y rows")
    U.assert_close(harness.to_host(buf.H_full()[ridx]), Hr, "bf16", "H rows")
    fs = f // p
    cols = np.array([0, fs - 1, fs, 2 * fs + 5, 3 * fs, f - 1], dtype=np.int64)   # shard boundaries
    dAc, dBr, db1c = orc.bwd_ffn_cols(X, A, b1, B, dZ, cols)
    cidx = torch.from_numpy(cols).cuda()
    U.assert_close(harness.to_host(buf.dA_full()[:, cidx]), dAc, "bf16", "dA cols")
    U.assert_close(harness.to_host(buf.dB_full()[cidx]), dBr, "bf16", "dB rows")
    U.assert_close(harness.to_host(buf.db1_sh.reshape(-1)[cidx]), db1c, "bf16", "db1")
    U.assert_close(harness.to_host(buf.db2), orc.bwd_db2(dZ), "bf16", "db2")
    xr = rows[-4:]
    U.assert_close(harness.to_host(buf.dX[torch.from_numpy(xr).cuda()]), orc.bwd_dX_rows(X, A, b1, B, dZ, xr),
                   "bf16", "dX rows")


def test_two_million_token_weight_gradients_sampled(env, orc):
    """s = 2^19, b = 4: M = 2^21 tokens, so the weight gradients contract over 32768 blocks of
    64 tokens.  In one accumulation the tensor cores' fp32 error alone reaches 2.5e-3 (rel.
    Frobenius) at this length; split into K chunks of 4096 blocks added in fp32 the sampled dA
    columns and dB rows meet the bf16 bound.  h = 128, ffn = 1024, p = 4 (Y, H, dH 4 GB each)."""
    import torch
    harness, synth, T = env
    assert T.tpmlp_get_k_chunk() == 4096
    wl = synth.custom(1 << 19, 4, 128, 1024, 4, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=2021)
    buf = harness.MLPBuffers(wl, backward=True)
    buf.fwd()
    buf.bwd()
    T.tpmlp_device_status()
    M, f, p = wl.M, wl.ffn, wl.p
    widen = synth.widen
    X, A, B = widen(buf.host["X"]), widen(buf.host["A"]), widen(buf.host["B"])
    b1, b2, dZ = widen(buf.host["b1"]), widen(buf.host["b2"]), widen(buf.host["dZ"])
    rows = np.array([0, 1, M // 2, M - 1], dtype=np.int64)
    Hr, Yr, Zr = orc.mlp_fwd(X[rows], A, b1, B, b2)
    U.assert_close(harness.to_host(buf.Z[torch.from_numpy(rows).cuda()]), Zr, "bf16", "Z rows")
    fs = f // p
    cols = np.array([0, fs - 1, fs, 2 * fs + 5, 3 * fs, f - 1], dtype=np.int64)
    dAc, dBr, db1c = orc.bwd_ffn_cols(X, A, b1, B, dZ, cols)
    cidx = torch.from_numpy(cols).cuda()
    U.assert_close(harness.to_host(buf.dA_full()[:, cidx]), dAc, "bf16", "dA cols")
    U.assert_close(harness.to_host(buf.dB_full()[cidx]), dBr, "bf16", "dB rows")
    U.assert_close(harness.to_host(buf.db1_sh.reshape(-1)[cidx]), db1c, "bf16", "db1")
    U.assert_close(harness.to_host(buf.db2), orc.bwd_db2(dZ), "bf16", "db2")


def test_last_wave_on_split_k_pairs(env, orc):
    """A shape whose six GEMMs all have more 256x256 tiles than CTA pairs, a last wave at most
    half full and K loops longer than 40 blocks (s=896 b=4 h=2568 ffn=5136 p=2: 308, 154 and 242
    tiles, remainders 4, 2 and 14 on 76 pairs), so in automatic mode every GEMM runs its full
    waves on CTA pairs and its last wave on split-K pairs of pairs.  Sampled rows and columns
    against the oracle (the last token rows lie in the last wave's tiles), and every element
    within fp32 reassociation of the same step on CTA pairs only (mode 3)."""
    import torch
    harness, synth, T = env
    wl = synth.custom(896, 4, 2568, 5136, 2, dtype="bf16", sigma_w=0.02, sigma_bias=0.05, seed=91)
    T.tpmlp_set_gemm_mode(3)
    try:
        ref = harness.MLPBuffers(wl, backward=True)
        ref.fwd()
        ref.bwd()
        T.tpmlp_set_gemm_mode(0)
        buf = harness.MLPBuffers(wl, backward=True, host=ref.host)
        buf.fwd()
        buf.bwd()
        T.tpmlp_device_status()
    finally:
        T.tpmlp_set_gemm_mode(0)
    for name, a, b in (("Z", buf.Z, ref.Z), ("dX", buf.dX, ref.dX), ("Y", buf.Y, ref.Y), ("dH", buf.dH, ref.dH)):
        err = float((a.double() - b.double()).norm() / b.double().norm())
        assert err < 2e-3, (name, err)
    for name, a, b in (("dA", buf.dA_sh, ref.dA_sh), ("dB", buf.dB_sh, ref.dB_sh)):
        err = float((a.double() - b.double()).norm() / b.double().norm())
        assert err < 1e-5, (name, err)
    M, h, f, p = wl.M, wl.h, wl.ffn, wl.p
    widen = synth.widen
    X, A, B, dZ = (widen(buf.host[k]) for k in ("X", "A", "B", "dZ"))
    b1, b2 = widen(buf.host["b1"]), widen(buf.host["b2"])
    rows = _rows(M, 6, 91)
    Hr, Yr, Zr = orc.mlp_fwd(X[rows], A, b1, B, b2)
    ridx = torch.from_numpy(rows).cuda()
    U.assert_close(harness.to_host(buf.Z[ridx]), Zr, "bf16", "Z rows")
    cols = _cols(f, p, 4, 91)
    dAc, dBr, db1c = orc.bwd_ffn_cols(X, A, b1, B, dZ, cols)
    cidx = torch.from_numpy(cols).cuda()
    U.assert_close(harness.to_host(buf.dA_full()[:, cidx]), dAc, "bf16", "dA cols")
    U.assert_close(harness.to_host(buf.dB_full()[cidx]), dBr, "bf16", "dB rows")
    xr = np.array([0, M // 2, M - 2, M - 1], dtype=np.int64)
    dXr = orc.bwd_dX_rows(X, A, b1, B, dZ, xr)
    U.assert_close(harness.to_host(buf.dX[torch.from_numpy(xr).cuda()]), dXr, "bf16", "dX rows")
