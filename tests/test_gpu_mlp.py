"""The MLP block through the C-ABI against the fp64 oracle on small shapes that
span several tiles and ragged tails in every GEMM dimension (GPU)."""
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


@pytest.fixture(params=[0, 1, 3, 4, 5], ids=["auto", "single-cta", "pair-direct", "pair-staged", "split-k"])
def gemm_mode(request, env):
    """The automatic tiling, or forced 128x256 single-CTA tiles, 256x256 CTA-pair tiles (either
    epilogue), or split-K CTA pairs for every shard-summing GEMM (row, dX) that fits one wave of
    them."""
    T = env[2]
    T.tpmlp_set_gemm_mode(request.param)
    yield request.param
    T.tpmlp_set_gemm_mode(0)


# (s, b, h, ffn, p): tiles are 128 (tokens) x 256 (outputs) x 64 (reduction)
SHAPES = [
    (25, 8, 72, 264, 3),      # M=200 ragged, h=72 ragged K, fs=88 ragged N
    (16, 8, 128, 512, 1),     # p = 1: the plain MLP
    (33, 4, 256, 1024, 2),    # M=132 (one row past a tile), fs=512 (two full N tiles)
    (64, 4, 320, 1280, 4),    # h=320: row GEMM N tail of 64, K of 5 blocks
    (7, 3, 512, 2048, 8),     # M=21, p=8
    (100, 3, 136, 544, 2),    # h=136 (2 K blocks + 8), fs=272 (256 + 16), M=300
    (128, 2, 192, 768, 6),    # p=6, fs=128
]


def _run_and_check(env, orc, wl, check_bwd=True):
    harness, synth, T = env
    buf = harness.MLPBuffers(wl, backward=check_bwd)
    # poison outputs so that unwritten elements show up as NaN
    for t in (buf.Z, buf.Y, buf.H):
        if t is not None:
            t.fill_(float("nan"))
    buf.fwd()
    if check_bwd:
        for t in (buf.dX, buf.dA_sh, buf.dB_sh, buf.db1_sh, buf.db2, buf.dH):
            t.fill_(float("nan"))
        buf.bwd()
    T.tpmlp_device_status()
    x = U.host_inputs_f64(buf)
    H, Y, Z = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    dt = wl.dtype
    U.assert_close(harness.to_host(buf.Z), Z, dt, "Z")
    U.assert_close(harness.to_host(buf.Y_full()), Y, dt, "Y")
    if buf.H is not None:
        U.assert_close(harness.to_host(buf.H_full()), H, dt, "H")
    if check_bwd:
        g = orc.mlp_bwd(x["X"], x["A"], x["B"], H, Y, x["dZ"])
        U.assert_close(harness.to_host(buf.dX), g["dX"], dt, "dX")
        U.assert_close(harness.to_host(buf.dA_full()), g["dA"], dt, "dA")
        U.assert_close(harness.to_host(buf.dB_full()), g["dB"], dt, "dB")
        U.assert_close(harness.to_host(buf.db1_sh).reshape(-1), g["db1"], dt, "db1")
        U.assert_close(harness.to_host(buf.db2), g["db2"], dt, "db2")
    return buf


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "s{}b{}h{}f{}p{}".format(*s))
def test_bf16_fwd_bwd_small(env, orc, shape, gemm_mode):
    _, synth, _ = env
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=sum(shape))
    _run_and_check(env, orc, wl)


def test_f32_tiny_workload(env, orc):
    """The tiny fp32 workload (s=8, b=2, h=64, ffn=256, p=2), forward and backward, <= 1e-5."""
    _, synth, _ = env
    _run_and_check(env, orc, synth.WORKLOADS[1])


@pytest.mark.parametrize("shape", [(5, 3, 48, 144, 3), (9, 7, 64, 256, 4)], ids=str)
def test_f32_small(env, orc, shape):
    _, synth, _ = env
    wl = synth.custom(*shape, dtype="f32", sigma_w=0.1, sigma_bias=0.1, seed=3)
    _run_and_check(env, orc, wl)


def test_every_divisor_p(env, orc, gemm_mode):
    """Sharded == unsharded for every legal p of one small problem (forward)."""
    _, synth, _ = env
    h, ffn = 96, 384
    for p in [d for d in range(1, 13) if ffn % d == 0 and h % d == 0 and (ffn // d) % 8 == 0]:
        wl = synth.custom(6, 11, h, ffn, p, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=5)
        _run_and_check(env, orc, wl, check_bwd=False)


def test_column_and_row_entry_points(env, orc, gemm_mode):
    """tpmlp_column_fwd (GeLU and identity) and tpmlp_row_fwd on their own."""
    import torch
    harness, synth, T = env
    wl = synth.custom(10, 13, 136, 528, 2, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=11)
    buf = harness.MLPBuffers(wl, backward=False)
    s, b, h, f, p = buf.dims()
    M, fs = s * b, f // p
    x = U.host_inputs_f64(buf)
    for act in (T.ACT_GELU_ERF, T.ACT_NONE):
        Y = torch.full((p, M, fs), float("nan"), dtype=torch.bfloat16, device="cuda")
        Hs = torch.full((p, M, fs), float("nan"), dtype=torch.bfloat16, device="cuda")
        T.tpmlp_column_fwd(buf.X, buf.A_sh, buf.b1_sh, Y, Hs, s, b, h, f, p, act=act)
        T.tpmlp_device_status()
        Href, Yref, _ = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], None,
                                    act=1 if act == T.ACT_GELU_ERF else 0)
        U.assert_close(harness.to_host(Y.permute(1, 0, 2).reshape(M, f)), Yref, "bf16", f"Y act={act}")
        U.assert_close(harness.to_host(Hs.permute(1, 0, 2).reshape(M, f)), Href, "bf16", f"H act={act}")
    # row layer alone on the GPU's own Y: Z = sum_i Y_i B_i + b2
    Z = torch.full((M, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_column_fwd(buf.X, buf.A_sh, buf.b1_sh, buf.Y, None, s, b, h, f, p)
    T.tpmlp_row_fwd(buf.Y, buf.B_sh, buf.b2, Z, s, b, h, f, p)
    T.tpmlp_device_status()
    Yg = harness.to_host(buf.Y_full())
    Zref = Yg @ x["B"] + x["b2"]
    U.assert_close(harness.to_host(Z), Zref, "bf16", "Z(row on GPU Y)")


def test_bias_added_once(env, orc):
    """With p = 4 a per-shard b2 would give Z + 3 b2: the oracle comparison catches it;
    here we also check Z(b2) - Z(0) == b2 exactly up to bf16 rounding."""
    import torch
    harness, synth, T = env
    wl = synth.custom(4, 8, 64, 256, 4, dtype="bf16", sigma_w=0.02, sigma_bias=0.5, seed=21)
    buf = harness.MLPBuffers(wl, backward=False)
    s, b, h, f, p = buf.dims()
    buf.fwd()
    Z0 = torch.empty_like(buf.Z)
    T.tpmlp_row_fwd(buf.Y, buf.B_sh, None, Z0, s, b, h, f, p)
    T.tpmlp_device_status()
    diff = harness.to_host(buf.Z) - harness.to_host(Z0)
    b2 = U.host_inputs_f64(buf)["b2"]
    assert np.max(np.abs(diff - b2)) < 0.02 * np.max(np.abs(b2)) + 0.02


def test_deterministic(env, orc, gemm_mode):
    harness, synth, T = env
    wl = synth.custom(50, 6, 256, 1024, 4, dtype="bf16", seed=2)
    buf = harness.MLPBuffers(wl, backward=True)
    buf.fwd()
    buf.bwd()
    first = [t.clone() for t in (buf.Z, buf.Y, buf.H, buf.dX, buf.dA_sh, buf.dB_sh, buf.db1_sh, buf.db2)]
    buf.fwd()
    buf.bwd()
    T.tpmlp_device_status()
    again = (buf.Z, buf.Y, buf.H, buf.dX, buf.dA_sh, buf.dB_sh, buf.db1_sh, buf.db2)
    import torch
    for a, b_ in zip(first, again):
        assert torch.equal(a, b_), "results differ between runs"


def test_guard_canaries(env, orc, gemm_mode):
    """Outputs written through pointers into the middle of larger buffers leave the
    surrounding guard bytes untouched."""
    import torch
    harness, synth, T = env
    wl = synth.custom(40, 5, 136, 544, 2, dtype="bf16", seed=8)
    buf = harness.MLPBuffers(wl, backward=True)
    s, b, h, f, p = buf.dims()
    M, fs = s * b, f // p
    G = 4096  # guard elements on each side (8 KiB)

    def guarded(n, dtype):
        big = torch.full((n + 2 * G,), 7.0, dtype=dtype, device="cuda")
        return big, big[G:G + n]

    zb, Z = guarded(M * h, torch.bfloat16)
    yb, Y = guarded(p * M * fs, torch.bfloat16)
    hb, Hs = guarded(p * M * fs, torch.bfloat16)
    T.tpmlp_mlp_fwd(buf.X, buf.A_sh, buf.b1_sh, buf.B_sh, buf.b2, Z, Y, Hs, s, b, h, f, p)
    xb, dX = guarded(M * h, torch.bfloat16)
    ab, dA = guarded(p * h * fs, torch.float32)
    bb, dB = guarded(p * fs * h, torch.float32)
    db1b, db1 = guarded(f, torch.float32)
    db2b, db2 = guarded(h, torch.float32)
    dhb, dH = guarded(p * M * fs, torch.bfloat16)
    T.tpmlp_mlp_bwd(buf.X, buf.A_sh, buf.B_sh, Hs, Y, buf.dZ, dX, dA, dB, db1, db2, dH, s, b, h, f, p)
    T.tpmlp_device_status()
    for big in (zb, yb, hb, xb, ab, bb, db1b, db2b, dhb):
        assert bool((big[:G] == 7.0).all()) and bool((big[-G:] == 7.0).all())
    # and the results equal the plain run
    buf.fwd()
    buf.bwd()
    T.tpmlp_device_status()
    assert bool((buf.Z.view(-1) == Z).all())
    assert bool((buf.dX.view(-1) == dX).all())


def test_empty_batch(env):
    import torch
    harness, synth, T = env
    dummy = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    out = torch.full((1024,), 3.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.full((1024,), 3.0, dtype=torch.bfloat16, device="cuda")
    assert T.tpmlp_mlp_fwd(dummy, dummy, None, dummy, None, out, ws, None, 0, 4, 64, 256, 2) == T.OK
    T.tpmlp_device_status()
    assert bool((out == 3.0).all()) and bool((ws == 3.0).all())


def test_single_and_pair_tiles_agree(env, orc):
    """Single-CTA and CTA-pair tiles accumulate in the same K order per element, and the two
    pair epilogues store the same values: results are bit-identical in every forced mode."""
    import torch
    harness, synth, T = env
    wl = synth.custom(150, 4, 384, 1536, 3, dtype="bf16", seed=9)
    buf = harness.MLPBuffers(wl, backward=True)
    out = {}
    for mode in (1, 2, 3, 4):
        T.tpmlp_set_gemm_mode(mode)
        buf.fwd()
        buf.bwd()
        T.tpmlp_device_status()
        out[mode] = [t.clone() for t in (buf.Z, buf.Y, buf.H, buf.dX, buf.dA_sh, buf.dB_sh, buf.dH)]
    T.tpmlp_set_gemm_mode(0)
    for mode in (2, 3, 4):
        for a, b_ in zip(out[1], out[mode]):
            assert torch.equal(a, b_), mode


@pytest.mark.parametrize("shape", [(40, 6, 192, 768, 3), (320, 8, 1024, 2048, 2)], ids=["narrow", "wide"])
def test_single_cta_tile_widths(env, orc, shape):
    """Single-CTA tiles are 128x128 when 128x256 tiles would leave more than half of the
    SMs idle, else 128x256.  The first shape runs every GEMM on 128x128 tiles; the second
    runs the column, row, dH and dX GEMMs on 128x256 tiles and dA, dB on 128x128."""
    _, synth, T = env
    T.tpmlp_set_gemm_mode(1)
    try:
        wl = synth.custom(*shape, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=sum(shape))
        _run_and_check(env, orc, wl)
    finally:
        T.tpmlp_set_gemm_mode(0)


@pytest.mark.parametrize("shape", [(10, 4, 256, 1024, 16), (6, 5, 512, 2048, 32)], ids=["p16", "p32"])
def test_many_shards(env, orc, shape, gemm_mode):
    """More shards than any page sizing uses (p = 16, 32; f/p = 64): the column GEMM has one
    narrow N-block per shard and the row / dX shard sums run 16-32 shards in one K loop."""
    _, synth, _ = env
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=sum(shape) + 3)
    _run_and_check(env, orc, wl)


@pytest.mark.parametrize("shape", [(1, 1, 8, 8, 1), (32, 1, 8, 64, 8), (1, 2, 16, 32, 2), (3, 1, 64, 8, 1),
                                   (1, 1, 64, 512, 1)],
                         ids=["one-token-h8", "h8-p8", "two-tokens", "fs8", "one-token-two-nblocks"])
def test_degenerate_shapes(env, orc, shape, gemm_mode):
    """The smallest legal problems: one token, h = 8 (one 16-byte row of X) with h / p = 1 and
    f / p = 8, every operand smaller than a single TMA box and a single tile in every GEMM (the
    last shape a single token over two 256-wide N-blocks).  The h = 8, p = 8 case runs 32 tokens: with one token its Z has 8 elements, too few
    for the relative Frobenius error to be more than a sample of the bf16 roundings (a CPU
    emulation of the kernels' rounding points, bf16 Y between the GEMMs and a bf16 Z store,
    gives 3.003e-3 there, exactly what the kernels produce).  One token also makes dA and dB
    outer products of bf16-rounded vectors, whose worst element carries one rounding unaveraged:
    at h = f = 512 the emulation exceeds the max-abs bound exactly as the kernels do, so the
    two-N-block case is 64 wide.  The emulation passes every shape here."""
    _, synth, _ = env
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.1, sigma_bias=0.05, seed=sum(shape) + 11)
    _run_and_check(env, orc, wl)


@pytest.mark.parametrize("shape", [(1, 1, 512, 512, 1), (1, 1, 8, 8, 1), (1, 2, 64, 512, 2), (1, 1, 1024, 4096, 4)],
                         ids=["one-token-h512", "one-token-h8", "two-tokens", "one-token-h1024"])
def test_tiny_outputs_elementwise_bound(env, orc, shape, gemm_mode):
    """The bound for outputs too small for the statistical ones (reading r8a): every element within
    the a-priori error of the rounding protocol (reading r7) of the exact values.  A bf16 rounding
    adds at most 2^-9 relative error; an fp32 sum of K terms at most K 2^-23 of the sum of
    magnitudes (2^-22 is used for margin); GeLU and GeLU' are 1.2-Lipschitz.  With u = half the
    bf16 spacing at the exact value, S = |dZ| |B|^T and s_X = |X| |A| (sums of magnitudes):
        eY  = 2^-8 |Y*| + 1.2 h 2^-22 s_X                        (Y from the fp32 H)
        eH  = 2^-9 |H*| + h 2^-22 s_X                            (the saved bf16 H)
        e   = (2^-8 |GeLU'(H*)| + 1.2 eH + |GeLU'(H*)| h 2^-22) S  (dH)
        |Z - Z*|   <= u(Z*) + eY |B| + f 2^-22 |Y*| |B|
        |dX - dX*| <= u(dX*) + e |A|^T + f 2^-22 |dH*| |A|^T
        |dA - dA*| <= |X|^T e + M 2^-22 |X|^T |dH*|,   |db1 - db1*| <= sum_m e + M 2^-22 sum_m |dH*|
        |dB - dB*| <= eY^T |dZ| + M 2^-22 |Y*|^T |dZ|
    The first shape is the one-token call whose weight gradients exceed the RMS-scaled max-abs
    bound by their own roundings."""
    from scipy.special import ndtr
    harness, synth, T = env
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.1, sigma_bias=0.05, seed=sum(shape) + 13)
    buf = harness.MLPBuffers(wl, backward=True)
    buf.fwd()
    buf.bwd()
    T.tpmlp_device_status()
    x = U.host_inputs_f64(buf)
    X, A, B, dZ = x["X"], x["A"], x["B"], x["dZ"]
    M, h = X.shape
    f = A.shape[1]
    H, Y, Z = orc.mlp_fwd(X, A, x["b1"], B, x["b2"])
    g = orc.mlp_bwd(X, A, B, H, Y, dZ)
    gp = ndtr(H) + H * np.exp(-0.5 * H * H) / np.sqrt(2.0 * np.pi)
    acc = 2.0 ** -22
    sX = np.abs(X) @ np.abs(A) + (0.0 if x["b1"] is None else np.abs(x["b1"]))
    S = np.abs(dZ) @ np.abs(B).T
    eY = 2.0 ** -8 * np.abs(Y) + 1.2 * h * acc * sX
    eH = 2.0 ** -9 * np.abs(H) + h * acc * sX
    e = (2.0 ** -8 * np.abs(gp) + 1.2 * eH + np.abs(gp) * h * acc) * S
    dHa = np.abs(gp) * S
    bounds = {
        "Z": (harness.to_host(buf.Z), Z,
              U.bf16_half_spacing(Z) + eY @ np.abs(B) + f * acc * (np.abs(Y) @ np.abs(B))),
        "dX": (harness.to_host(buf.dX), g["dX"],
               U.bf16_half_spacing(g["dX"]) + e @ np.abs(A).T + f * acc * (dHa @ np.abs(A).T)),
        "dA": (harness.to_host(buf.dA_full()), g["dA"], np.abs(X).T @ e + M * acc * (np.abs(X).T @ dHa)),
        "dB": (harness.to_host(buf.dB_full()), g["dB"], eY.T @ np.abs(dZ) + M * acc * (np.abs(Y).T @ np.abs(dZ))),
        "db1": (harness.to_host(buf.db1_sh).reshape(-1), g["db1"], e.sum(axis=0) + M * acc * dHa.sum(axis=0)),
    }
    for name, (got, ref, bound) in bounds.items():
        excess = np.abs(got - ref) - (bound + 1e-7)
        assert float(np.max(excess)) <= 0.0, f"{name}: {float(np.max(excess)):.3e} beyond the element bound"


def test_mixed_wave_shape(env, orc):
    """A shape whose row and dX GEMMs have 80 pair tiles (76 pairs fit at once), so the
    last wave holds 4 tiles, which walk K (and the shard sum) backwards; the
    weight-gradient GEMMs have fewer tiles than pairs."""
    _, synth, _ = env
    wl = synth.custom(320, 8, 2048, 1024, 2, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=77)
    _run_and_check(env, orc, wl)


@pytest.mark.parametrize("mode", [3, 4], ids=["pair-direct", "pair-staged"])
def test_every_gemm_two_waves(env, orc, mode):
    """All six GEMMs with more pair tiles than co-resident pairs (80 to 100 tiles), so
    every GEMM has second-wave tiles that walk K backwards: the batched column, dH,
    dA and dB GEMMs as well as the shard-summing row and dX GEMMs.  Full parity, with
    either epilogue of the pair kernel."""
    _, synth, T = env
    T.tpmlp_set_gemm_mode(mode)
    try:
        wl = synth.custom(512, 4, 2560, 2560, 2, dtype="bf16", sigma_w=0.02, sigma_bias=0.05, seed=78)
        _run_and_check(env, orc, wl)
    finally:
        T.tpmlp_set_gemm_mode(0)


@pytest.mark.parametrize("mode", [1, 3], ids=["single-cta", "pair-direct"])
def test_split_contraction(env, orc, mode):
    """Weight gradients split into K chunks of 64 and 128 tokens (M = 200: four and two
    launches, the last one ragged), each later launch adding its partial product to the fp32
    dA / dB: full parity, and within fp32 rounding of the unsplit run (the other outputs are
    bit-identical: only fp32-output contractions are split)."""
    import torch
    harness, synth, T = env
    T.tpmlp_set_gemm_mode(mode)
    try:
        wl = synth.custom(50, 4, 320, 2048, 2, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=80)
        whole = _run_and_check(env, orc, wl)
        ref = [t.clone() for t in (whole.Z, whole.dX, whole.dA_sh, whole.dB_sh, whole.dH)]
        for chunk in (1, 2):
            T.tpmlp_set_k_chunk(chunk)
            buf = _run_and_check(env, orc, wl)
            assert torch.equal(buf.Z, ref[0]) and torch.equal(buf.dX, ref[1]) and torch.equal(buf.dH, ref[4])
            for got, want in ((buf.dA_sh, ref[2]), (buf.dB_sh, ref[3])):
                err = (got.double() - want.double()).norm() / want.double().norm()
                assert float(err) < 1e-6, float(err)
    finally:
        T.tpmlp_set_k_chunk(0)
        T.tpmlp_set_gemm_mode(0)


@pytest.mark.parametrize("shape", [(60, 5, 264, 576, 3), (256, 4, 1024, 4096, 4), (130, 3, 520, 2080, 2)],
                         ids=["odd-k-blocks", "s256-h1024", "ragged"])
def test_split_k_tiles(env, orc, shape):
    """Split-K CTA pairs (mode 5) on the row and dX GEMMs: two pairs of a cluster each sum half
    of the K blocks and add their partials through distributed shared memory.  Shard counts and
    widths make the split fall inside a shard (3 shards x 3 K blocks: the halves are 4 and 5
    blocks), on a workload-sized K loop (64 blocks), and on ragged M, N and K.  Full parity with
    the oracle, and within fp32 reassociation of the CTA-pair result."""
    import torch
    harness, synth, T = env
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.03, sigma_bias=0.05, seed=sum(shape) + 5)
    T.tpmlp_set_gemm_mode(3)
    try:
        ref = _run_and_check(env, orc, wl)
        want = [t.clone() for t in (ref.Z, ref.dX)]
        T.tpmlp_set_gemm_mode(5)
        buf = _run_and_check(env, orc, wl)
    finally:
        T.tpmlp_set_gemm_mode(0)
    for got, w in zip((buf.Z, buf.dX), want):
        err = (got.double() - w.double()).norm() / w.double().norm()
        assert float(err) < 2e-3, float(err)


def _random_shapes(n, seed):
    """Random (s, b, h, ffn, p) with h % p == 0, h % 8 == 0 and ffn/p % 8 == 0."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        p = int(rng.choice([1, 2, 3, 4, 5, 6, 8]))
        step = 8 * p // int(np.gcd(8, p))          # lcm(8, p)
        h = step * int(rng.integers(1, 600 // step + 1))
        fs = 8 * int(rng.integers(1, 65))
        s, b = int(rng.integers(1, 40)), int(rng.integers(1, 9))
        if fs * p > 3000:
            continue
        out.append((s, b, h, fs * p, p))
    return out


@pytest.mark.parametrize("shape", _random_shapes(12, 2026), ids=lambda s: "s{}b{}h{}f{}p{}".format(*s))
def test_random_shapes(env, orc, shape, gemm_mode):
    """Random small shapes (token counts, widths and shard counts off every tile boundary)."""
    _, synth, _ = env
    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=sum(shape) + 1)
    _run_and_check(env, orc, wl)
