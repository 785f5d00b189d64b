"""The kernels round where reading r7 of the tolerance says they do (GPU).

Reading r7 fixes the precision of every intermediate: fp32 accumulation, H = XA + b1 in fp32,
Y = GeLU(H) from that fp32 H rounded to bf16, H stored as bf16, Z = YB + b2 rounded to bf16;
dH = (dZ Bᵀ) · GeLU'(H) from the stored bf16 H, rounded to bf16; dX = dH Aᵀ rounded to bf16;
dA = Xᵀ dH, dB = Yᵀ dZ and db1 = 1ᵀdH in fp32 from the bf16 dH and Y.  This file builds those
steps on the CPU (numpy in fp64, scipy's erfc, torch's CPU bf16 rounding, nothing from the CUDA
path) and compares the kernels' outputs with them element by element.  The two differ only
through fp32 accumulation order and the kernels' erfc approximation (|error| <= 1.5e-7), which
move a bf16 rounding by one unit where the exact value sits that close to a rounding boundary:
a small fraction of the elements, never more than one unit.  A different rounding protocol
(GeLU of the bf16 H, GeLU' of an fp32 H, a missing or doubled rounding) changes a large
fraction of the elements, which the tolerance against the fp64 oracle cannot tell apart.
"""
import numpy as np
import pytest
from scipy import special

import gpu_util as U

pytestmark = pytest.mark.gpu

# At most this fraction of a bf16 tensor's elements may differ from the emulation, each by one
# bf16 unit.  The expected fraction is about 2 * (relative fp32 error) * 2^8 per element: below
# 0.2 % for the sums of a few thousand terms here.
MAX_FLIP_FRACTION = 0.01
# Outputs computed from an earlier bf16 stage (Z from Y; dX, dA, db1 from dH; dB from Y): the
# earlier stage's one-unit differences propagate, giving a relative Frobenius difference of
# about sqrt(flip fraction) * 2^-8 (1-2e-4 at the fractions expected here).  A rounding out of
# place (a bias added after a bf16 rounding, a second rounding) adds ~1e-3, a third of the
# tolerance against the fp64 oracle.
REL_F_DOWNSTREAM = 1e-3


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth, tpmlp
    return harness, synth, tpmlp


def _bf16(a):
    """Round to bf16, nearest even (torch's CPU conversion), returned as fp64."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).bfloat16().double().numpy()


def _f32(a):
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _gelu(x):
    return x * 0.5 * special.erfc(-x / np.sqrt(2.0))


def _gelu_grad(x):
    return 0.5 * special.erfc(-x / np.sqrt(2.0)) + x * np.exp(-0.5 * x * x) / np.sqrt(2.0 * np.pi)


def _emulate(X, A, b1, B, b2, dZ, gelu_of_saved_h=False, grad_of_fp32_h=False):
    """The rounding points of reading r7 on exact (fp64) sums.  The two flags build the
    plausible wrong protocols that the host test shows this comparison tells apart."""
    Hf = _f32(X @ A + b1)              # fp32 pre-activation
    H = _bf16(Hf)                       # the saved pre-activation
    Y = _bf16(_gelu(H if gelu_of_saved_h else Hf))  # GeLU of the fp32 value
    Z = _bf16(Y @ B + b2)
    dY = _f32(dZ @ B.T)
    dH = _bf16(dY * _gelu_grad(Hf if grad_of_fp32_h else H))  # GeLU' of the stored bf16 H
    dX = _bf16(dH @ A.T)
    return {"H": H, "Y": Y, "Z": Z, "dH": dH, "dX": dX,
            "dA": X.T @ dH, "dB": Y.T @ dZ, "db1": dH.sum(0), "db2": dZ.sum(0)}


def _flip_fraction(got, emu, name):
    """The fraction of a bf16 tensor's elements that differ from the emulation, bounded."""
    assert got.shape == emu.shape, (name, got.shape, emu.shape)
    assert U.stored_as_bf16(got), f"{name}: not bf16 values"
    flips = float(np.mean(got != emu))
    assert flips <= MAX_FLIP_FRACTION, f"{name}: {100 * flips:.2f} % of elements differ from the emulation"
    return flips


def _check_bf16(got, emu, name, floor_frac=2.0 ** -10):
    """Every element equal to the emulation or one bf16 unit away; few of them away.  Units
    are measured at max(|value|, 2^-10 RMS): where a sum nearly cancels, the absolute error of
    fp32 accumulation (a few 1e-7 of the terms here) exceeds the tiny result's own bf16 unit,
    whatever the rounding protocol."""
    assert got.shape == emu.shape, (name, got.shape, emu.shape)
    assert U.stored_as_bf16(got), f"{name}: not bf16 values"
    floor = floor_frac * float(np.sqrt(np.mean(emu * emu)))
    unit = 2.0 * U.bf16_half_spacing(np.maximum(np.maximum(np.abs(got), np.abs(emu)), floor))
    units = np.abs(got - emu) / unit
    assert float(np.max(units)) <= 1.0, f"{name}: {float(np.max(units)):.1f} bf16 units from the emulation"
    return _flip_fraction(got, emu, name)


@pytest.mark.parametrize("mode", [1, 3, 4, 5], ids=["single-cta", "pair-direct", "pair-staged", "split-k"])
def test_rounding_points_match_emulation(env, mode):
    harness, synth, T = env
    T.tpmlp_set_gemm_mode(mode)
    try:
        wl = synth.custom(64, 4, 512, 2048, 4, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=96)
        buf = harness.MLPBuffers(wl, backward=True)
        buf.fwd()
        buf.bwd()
        T.tpmlp_device_status()
    finally:
        T.tpmlp_set_gemm_mode(0)
    x = U.host_inputs_f64(buf)
    emu = _emulate(x["X"], x["A"], x["b1"], x["B"], x["b2"], x["dZ"])
    M, f = wl.M, wl.ffn
    # the stage whose inputs are exact: element by element, in bf16 units
    flips = {k: _check_bf16(harness.to_host(t), emu[k], k) for k, t in (("H", buf.H_full()), ("Y", buf.Y_full()))}
    # dH takes GeLU' of the saved H, so H's one-unit differences reach it, and near GeLU's
    # inflection (GeLU'(h) = 0 at h = -0.752) one unit of H moves GeLU' by ~1e-3 absolute, many
    # units of a small dH: its elements are counted, not bounded one by one
    dH = harness.to_host(buf.dH.permute(1, 0, 2).reshape(M, f))
    flips["dH"] = _flip_fraction(dH, emu["dH"], "dH")
    # stages fed by an earlier bf16 stage
    rel = {"dH": float(np.linalg.norm(dH - emu["dH"]) / np.linalg.norm(emu["dH"]))}
    assert rel["dH"] <= REL_F_DOWNSTREAM, f"dH: rel Frobenius {rel['dH']:.2e} from the emulation"
    for k, t in (("Z", buf.Z), ("dX", buf.dX), ("dA", buf.dA_full()), ("dB", buf.dB_full()),
                 ("db1", buf.db1_sh.reshape(-1)), ("db2", buf.db2)):
        g = harness.to_host(t)
        rel[k] = float(np.linalg.norm(g - emu[k]) / np.linalg.norm(emu[k]))
        assert rel[k] <= REL_F_DOWNSTREAM, f"{k}: rel Frobenius {rel[k]:.2e} from the emulation"
    print("one-unit fraction:", {k: f"{v:.2e}" for k, v in flips.items()},
          "rel. Frobenius from the emulation:", {k: f"{v:.1e}" for k, v in rel.items()})


# ---------------------------------------------------------------------------- SwiGLU (reading r14)
def _silu(x):
    return x * special.expit(x)


def _silu_grad(x):
    s = special.expit(x)
    return s * (1.0 + x * (1.0 - s))


def _emulate_swiglu(X, G, Uw, bg, bu, B, b2, dZ, bf16_saves=False):
    """Reading r14's rounding points: fp32 gate and up pre-activations (saved in fp32),
    Y = bf16(silu(g) u), Z = bf16(Y B + b2); dY in fp32, dg = bf16(dY u silu'(g)),
    du = bf16(dY silu(g)), dX = bf16(dg Gᵀ + du Uᵀ); fp32 weight and bias gradients."""
    Hg, Hu = _f32(X @ G + bg), _f32(X @ Uw + bu)
    Y = _bf16(_silu(Hg) * Hu)
    Z = _bf16(Y @ B + b2)
    dY = _f32(dZ @ B.T)
    if bf16_saves:  # the wrong protocol the host test separates: pre-activations saved in bf16
        Hg, Hu = _bf16(Hg), _bf16(Hu)
    dHg, dHu = _bf16(dY * Hu * _silu_grad(Hg)), _bf16(dY * _silu(Hg))
    return {"Hg": Hg, "Hu": Hu, "Y": Y, "Z": Z, "dHg": dHg, "dHu": dHu, "dX": _bf16(dHg @ G.T + dHu @ Uw.T),
            "dG": X.T @ dHg, "dU": X.T @ dHu, "dB": Y.T @ dZ, "dbg": dHg.sum(0), "dbu": dHu.sum(0),
            "db2": dZ.sum(0)}


@pytest.mark.parametrize("mode", [1, 2], ids=["single-cta", "cta-pair"])
def test_swiglu_rounding_points_match_emulation(env, orc, mode):
    import torch
    harness, synth, T = env
    s, b, h, f, p = 64, 4, 512, 2048, 4
    M, fs = s * b, f // p
    gen = lambda stream, shp, sig: synth.normal(97, stream, shp, sig, "bf16")  # noqa: E731
    X, G, Uw, B = gen(1, (M, h), 1.0), gen(2, (h, f), 0.05), gen(9, (h, f), 0.05), gen(3, (f, h), 0.05)
    bg, bu, b2, dZ = gen(4, (f,), 0.05), gen(10, (f,), 0.05), gen(5, (h,), 0.05), gen(6, (M, h), 1.0)
    d = harness.to_torch
    T.tpmlp_set_gemm_mode(mode)
    try:
        W = torch.empty((p, h, 2 * fs), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_swiglu_pack(d(G), d(Uw), W, h, f, p)
        bw = torch.empty((p, 2 * fs), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_swiglu_pack(d(bg), d(bu), bw, 1, f, p)
        Bd = d(B).view(p, fs, h)
        Z = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
        Y = torch.empty((p, M, fs), dtype=torch.bfloat16, device="cuda")
        H = torch.empty((p, M, 2 * fs), dtype=torch.float32, device="cuda")
        T.tpmlp_swiglu_mlp_fwd(d(X), W, bw, Bd, d(b2), Z, Y, H, s, b, h, f, p)
        dX = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
        dW = torch.empty((p, h, 2 * fs), dtype=torch.float32, device="cuda")
        dB = torch.empty((p, fs, h), dtype=torch.float32, device="cuda")
        dbw = torch.empty((p, 2 * fs), dtype=torch.float32, device="cuda")
        db2 = torch.empty((h,), dtype=torch.float32, device="cuda")
        dH = torch.empty((p, M, 2 * fs), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_swiglu_mlp_bwd(d(X), W, Bd, H, Y, d(dZ), dX, dW, dB, dbw, db2, dH, s, b, h, f, p)
        T.tpmlp_device_status()
    finally:
        T.tpmlp_set_gemm_mode(0)
    x = synth.widen
    emu = _emulate_swiglu(x(X), x(G), x(Uw), x(bg), x(bu), x(B), x(b2), x(dZ))
    host = harness.to_host
    Hg, Hu = orc.swiglu_unpack(host(H.permute(1, 0, 2)).transpose(1, 0, 2).copy(), p)
    for k, v in (("Hg", Hg), ("Hu", Hu)):  # saved in fp32: the fp32 sums themselves
        assert np.max(np.abs(v - emu[k])) <= 1e-5 * max(1.0, float(np.max(np.abs(emu[k])))), k
    dHg, dHu = orc.swiglu_unpack(host(dH), p)
    # stages whose inputs are fp32 sums: element by element, in bf16 units
    flips = {k: _check_bf16(v, emu[k], k)
             for k, v in (("Y", host(Y.permute(1, 0, 2).reshape(M, f))), ("dHg", dHg), ("dHu", dHu))}
    dG, dU = orc.swiglu_unpack(host(dW), p)
    dbg, dbu = orc.swiglu_unpack(host(dbw).reshape(p, 1, 2 * fs), p)
    rel = {}
    for k, v in (("Z", host(Z)), ("dX", host(dX)), ("dG", dG), ("dU", dU), ("dB", host(dB.reshape(f, h))),
                 ("dbg", dbg.reshape(-1)), ("dbu", dbu.reshape(-1)), ("db2", host(db2))):
        rel[k] = float(np.linalg.norm(v - emu[k]) / np.linalg.norm(emu[k]))
        assert rel[k] <= REL_F_DOWNSTREAM, f"{k}: rel Frobenius {rel[k]:.2e} from the emulation"
    print("one-unit fraction:", {k: f"{v:.2e}" for k, v in flips.items()},
          "rel. Frobenius from the emulation:", {k: f"{v:.1e}" for k, v in rel.items()})


@pytest.mark.parametrize("wi", [5, 4], ids=["fwd-bwd-s2048-b4-h5120", "fwd-s4096-b1-h8192"])
def test_full_workload_rounding_points_sampled(env, wi):
    """The bench's fwd+bwd workload (s=2048 b=4 h=5120 f=20480 p=4), and the forward at the
    pages' sizing (s=4096 b=1 h=8192 f=32768 p=8, K = 8192 and 32768), in their own launch
    configuration (multi-wave pair tiles walking K backwards), on 16 sampled token rows: H, Y, Z, dH and dX are row-local, so the emulation of
    reading r7 needs only those rows and the full weights.  With K = 5120 and 20480 the fp32
    accumulation error (measured ~1.9e-8 per 16-deep MMA step, growing linearly) reaches ~1e-5
    of the partial sums, so units are measured at max(|value|, RMS / 16), where it stays below
    0.05 unit; the expected fraction of one-unit differences is ~0.3-0.5 % (bound 1 %).
    Downstream, the K = 20480-32768 sums of Z and dX flip 1-2 % of their own roundings on
    accumulation order alone (~4-6e-4 relative) on top of the propagated flips (~2.5e-4): bound
    2e-3, which is below the
    3e-3 bar against the oracle; the flip fractions are what tell a wrong protocol (~25 %)."""
    harness, synth, T = env
    wl = synth.WORKLOADS[wi]
    buf = harness.MLPBuffers(wl, backward=True)  # with the H save; the backward runs only if the workload has one
    buf.fwd()
    if wl.backward:
        buf.bwd()
    T.tpmlp_device_status()
    M, f = wl.M, wl.ffn
    rng = np.random.default_rng(5)
    rows = np.array(sorted({0, M - 1} | set(rng.integers(0, M, 14).tolist())), dtype=np.int64)
    x = U.host_inputs_f64(buf)
    X, A, B = x["X"][rows], x["A"], x["B"]
    b1 = 0.0 if x["b1"] is None else x["b1"]
    b2 = 0.0 if x["b2"] is None else x["b2"]
    Hf = _f32(X @ A + b1)
    H = _bf16(Hf)
    Y = _bf16(_gelu(Hf))
    emu = {"H": H, "Y": Y, "Z": _bf16(Y @ B + b2)}
    import torch
    ridx = torch.from_numpy(rows).cuda()
    got = {"H": buf.H_full()[ridx], "Y": buf.Y_full()[ridx], "Z": buf.Z[ridx]}
    if wl.backward:
        dH = _bf16(_f32(x["dZ"][rows] @ B.T) * _gelu_grad(H))
        emu.update(dH=dH, dX=_bf16(dH @ A.T))
        got.update(dH=buf.dH.permute(1, 0, 2).reshape(M, f)[ridx], dX=buf.dX[ridx])
    got = {k: harness.to_host(v) for k, v in got.items()}
    flips = {k: _check_bf16(got[k], emu[k], k, floor_frac=2.0 ** -4) for k in ("H", "Y")}
    if wl.backward:
        flips["dH"] = _flip_fraction(got["dH"], emu["dH"], "dH")
    rel = {}
    for k in [k for k in ("dH", "Z", "dX") if k in emu]:
        rel[k] = float(np.linalg.norm(got[k] - emu[k]) / np.linalg.norm(emu[k]))
        assert rel[k] <= 2e-3, f"{k}: rel Frobenius {rel[k]:.2e} from the emulation"
    print("one-unit fraction:", {k: f"{v:.2e}" for k, v in flips.items()},
          "rel. Frobenius from the emulation:", {k: f"{v:.1e}" for k, v in rel.items()})


# ---------------------------------------------------------------------- attention projections
@pytest.mark.parametrize("mode", [1, 3, 4], ids=["single-cta", "pair-direct", "pair-staged"])
def test_attention_projection_rounding_points(env, orc, mode):
    """QKV = bf16(X W + b) over the per-head interleave, Z = bf16(ctx W_o + b_o) summed over the
    ranks' head blocks, dctx = bf16(dZ W_oᵀ), dX = bf16(dQKV Wᵀ) summed over ranks: each a single
    rounding of an fp32 sum of exact inputs, so every element is checked in bf16 units; the fp32
    weight and bias gradients have no bf16 stage before them (rel. Frobenius <= 1e-5)."""
    import torch
    harness, synth, T = env
    s, b, h, heads, p = 64, 4, 512, 8, 4
    M, hq = s * b, 3 * h // p
    gen = lambda stream, shp, sig: synth.normal(98, stream, shp, sig, "bf16")  # noqa: E731
    X, Wq, bq = gen(1, (M, h), 1.0), gen(2, (h, 3 * h), 0.05), gen(4, (3 * h,), 0.05)
    dQ, ctx, Wo, bo, dZ = gen(6, (M, 3 * h), 1.0), gen(7, (M, h), 1.0), gen(3, (h, h), 0.05), gen(5, (h,), 0.05), \
        gen(8, (M, h), 1.0)
    d, host, x = harness.to_torch, harness.to_host, synth.widen
    T.tpmlp_set_gemm_mode(mode)
    try:
        Wi = torch.empty((h, 3 * h), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_qkv_interleave(d(Wq), Wi, h, h, heads, p)
        bi = torch.empty((3 * h,), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_qkv_interleave(d(bq), bi, 1, h, heads, p)
        W_sh = torch.empty((p, h, hq), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_shard_columns(Wi, W_sh, h, 3 * h, p)
        QKV = torch.empty((p, M, hq), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_column_fwd(d(X), W_sh, bi, QKV, None, s, b, h, 3 * h, p, act=T.ACT_NONE)
        dQd = d(dQ).view(M, p, hq).permute(1, 0, 2).contiguous()
        dX = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
        dW = torch.empty((p, h, hq), dtype=torch.float32, device="cuda")
        db = torch.empty((p, hq), dtype=torch.float32, device="cuda")
        T.tpmlp_column_bwd(d(X), W_sh, dQd, dX, dW, db, s, b, h, 3 * h, p)
        ctx_sh = d(ctx).view(M, p, h // p).permute(1, 0, 2).contiguous()
        Z = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_row_fwd(ctx_sh, d(Wo), d(bo), Z, s, b, h, h, p)
        dctx = torch.empty((p, M, h // p), dtype=torch.bfloat16, device="cuda")
        dWo = torch.empty((p, h // p, h), dtype=torch.float32, device="cuda")
        dbo = torch.empty((h,), dtype=torch.float32, device="cuda")
        T.tpmlp_row_bwd(ctx_sh, d(Wo), d(dZ), None, dctx, dWo, dbo, s, b, h, h, p, act=T.ACT_NONE)
        T.tpmlp_device_status()
    finally:
        T.tpmlp_set_gemm_mode(0)
    Wih = orc.qkv_interleave(x(Wq), h, heads)          # layout map only
    bih = orc.qkv_interleave(x(bq)[None, :], h, heads)[0]
    Xf, dQf, ctxf, Wof, dZf = x(X), x(dQ), x(ctx), x(Wo), x(dZ)
    bf16_out = {"QKV": (host(QKV.permute(1, 0, 2).reshape(M, 3 * h)), _bf16(_f32(Xf @ Wih + bih))),
                "dX": (host(dX), _bf16(_f32(dQf @ Wih.T))),
                "Z": (host(Z), _bf16(_f32(ctxf @ Wof + x(bo)))),
                "dctx": (host(dctx.permute(1, 0, 2).reshape(M, h)), _bf16(_f32(dZf @ Wof.T)))}
    flips = {k: _check_bf16(g, e, k) for k, (g, e) in bf16_out.items()}
    for k, g, e in (("dW", host(dW.permute(1, 0, 2).reshape(h, 3 * h)), Xf.T @ dQf), ("db", host(db.reshape(-1)), dQf.sum(0)),
                    ("dWo", host(dWo.reshape(h, h)), ctxf.T @ dZf), ("dbo", host(dbo), dZf.sum(0))):
        err = float(np.linalg.norm(g - e) / np.linalg.norm(e))
        assert err <= 1e-5, f"{k}: rel Frobenius {err:.2e} from the exact sum"
    print("one-unit fraction:", {k: f"{v:.2e}" for k, v in flips.items()})
