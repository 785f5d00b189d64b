"""Pins of the oracle to facts the pages and mathematics fix (not to itself).

Each ``pin_*`` takes a loaded ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with the fact.  ``test_oracle_pins.py`` runs them on the
committed oracle; ``test_oracle_mutants.py`` runs them on builds with planted
mistakes and expects at least one to fail for each mistake.

Passages (web pages on Megatron tensor parallelism):
  [CP] "列并行" article (aiqz.cc): 切分原理, 数学基础, MLP 应用, Python 演示
  [M2] "Megatron 专家面试题 Level 2" (blog.cptz.space): M025, M026, M030
  [DP] "分布式并行训练全景" (talentme.airsota.com): 考点 2, 第三章 NumPy demo
"""
from __future__ import annotations

import math

import numpy as np
from scipy import special, stats

import oracle as _o


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(seed, M, h, f, bias=True, wscale=0.3):
    r = _rng(seed)
    X = r.standard_normal((M, h))
    A = r.standard_normal((h, f)) * wscale
    B = r.standard_normal((f, h)) * wscale
    b1 = r.standard_normal(f) * 0.1 if bias else None
    b2 = r.standard_normal(h) * 0.1 if bias else None
    dZ = r.standard_normal((M, h))
    return X, A, b1, B, b2, dZ


def _divisors(n):
    return [d for d in range(1, n + 1) if n % d == 0]


# --------------------------------------------------------------------------
# GeLU: the definition z * Phi(z) ([CP] MLP 应用, GeLU 定义)

def pin_gelu_closed_forms(orc):
    assert orc.gelu(0.0) == 0.0
    assert abs(orc.gelu_grad(0.0) - 0.5) < 1e-15
    # Phi(1) from a normal table: 0.841344746068543; Phi(-1) = 1 - Phi(1)
    assert abs(orc.gelu(1.0) - 0.8413447460685429) < 1e-15
    assert abs(orc.gelu(-1.0) + 0.15865525393145707) < 1e-15
    # Phi(x) + Phi(-x) = 1  =>  GeLU(x) - GeLU(-x) = x
    for x in (0.1, 0.7, 1.3, 2.9, 5.0, 11.0):
        assert abs((orc.gelu(x) - orc.gelu(-x)) - x) < 1e-14 * max(1.0, x)
    # tails: GeLU(x)/x -> 1 for large x, GeLU(-x) -> 0
    assert abs(orc.gelu(12.0) / 12.0 - 1.0) < 1e-15
    assert abs(orc.gelu(-12.0)) < 1e-30
    # GeLU' = 1 / 0 in the tails
    assert abs(orc.gelu_grad(12.0) - 1.0) < 1e-15 and abs(orc.gelu_grad(-12.0)) < 1e-28


def pin_gelu_vs_library(orc):
    """Against scipy's normal CDF/PDF (an independent library) and a finite difference."""
    xs = np.linspace(-8.0, 8.0, 321)
    for x in xs:
        ref = x * special.ndtr(x)
        assert abs(orc.gelu(x) - ref) <= 1e-15 * max(1.0, abs(ref)) + 1e-300
        refd = special.ndtr(x) + x * stats.norm.pdf(x)
        assert abs(orc.gelu_grad(x) - refd) <= 2e-15
        eps = 1e-5
        fd = (orc.gelu(x + eps) - orc.gelu(x - eps)) / (2 * eps)
        assert abs(orc.gelu_grad(x) - fd) < 1e-9


# --------------------------------------------------------------------------
# Column-parallel first layer ([CP] 数学基础 / 切分原理; [M2] M025)

def pin_column_concatenation_bitexact(orc):
    """X [A_1 || ... || A_p] == [X A_1 || ... || X A_p], bit for bit, every divisor p (incl. 3)."""
    M, h, f = 5, 7, 24
    X, A, b1, B, _, _ = _problem(1, M, h, f)
    H, Y, _ = orc.mlp_fwd(X, A, b1, B, None)
    for p in _divisors(f):
        fs = f // p
        parts_H, parts_Y = [], []
        for i in range(p):
            Ai = np.ascontiguousarray(A[:, i * fs:(i + 1) * fs])
            Bi = np.ascontiguousarray(B[i * fs:(i + 1) * fs, :])
            Hi, Yi, _ = orc.mlp_fwd(X, Ai, b1[i * fs:(i + 1) * fs], Bi, None)
            parts_H.append(Hi)
            parts_Y.append(Yi)
        # column identity and GeLU split invariance ([CP] MLP 应用, 分块不变性)
        assert np.array_equal(np.concatenate(parts_H, axis=1), H)
        assert np.array_equal(np.concatenate(parts_Y, axis=1), Y)


def pin_column_vs_numpy_demo(orc):
    """The [CP] Python 演示 setup (batch 4, d_in 8, d_out 9, p 3): per-shard X@W_i,
    concatenated, equals X@W; and the oracle's H equals numpy's X@W (independent matmul)."""
    r = _rng(42)
    X = r.standard_normal((4, 8))
    W = r.standard_normal((8, 9))
    shards = np.split(W, 3, axis=1)
    Ycat = np.concatenate([X @ Wi for Wi in shards], axis=1)
    H, _, _ = orc.mlp_fwd(X, W, None, np.zeros((9, 8)), None, act=_o.ACT_NONE)
    assert np.allclose(Ycat, X @ W)
    assert np.max(np.abs(H - X @ W)) <= 1e-13 * np.max(np.abs(X @ W))


# --------------------------------------------------------------------------
# Row-parallel second layer and the shard sum ([M2] M026; [DP] 考点 2)

def pin_row_sum_equals_unsharded(orc):
    """sum_i GeLU(X A_i + b1_i) B_i + b2 == oracle(X, A, B) for every divisor p; b2 once."""
    M, h, f = 6, 8, 36
    X, A, b1, B, b2, _ = _problem(2, M, h, f)
    _, _, Z = orc.mlp_fwd(X, A, b1, B, b2)
    for p in _divisors(f):
        fs = f // p
        acc = np.zeros((M, h))
        for i in range(p):
            sl = slice(i * fs, (i + 1) * fs)
            _, _, Zi = orc.mlp_fwd(X, np.ascontiguousarray(A[:, sl]), b1[sl],
                                   np.ascontiguousarray(B[sl, :]), None)
            acc += Zi
        acc += b2
        assert np.max(np.abs(acc - Z)) <= 1e-12 * np.max(np.abs(Z))


def pin_identity_activation_vs_numpy(orc):
    """With the identity in place of GeLU the block is the affine map (X A + b1) B + b2."""
    M, h, f = 9, 12, 20
    X, A, b1, B, b2, _ = _problem(3, M, h, f)
    H, Y, Z = orc.mlp_fwd(X, A, b1, B, b2, act=_o.ACT_NONE)
    ref = (X @ A + b1) @ B + b2
    assert np.max(np.abs(Z - ref)) <= 1e-12 * np.max(np.abs(ref))
    assert np.max(np.abs(H - (X @ A + b1))) <= 1e-12 * np.max(np.abs(H))


def pin_relu_demo_structure(orc):
    """The [DP] 第三章 NumPy demo (x 2x8, w1 8x32, w2 32x8, tp 2, ReLU stand-in):
    per-rank maximum(0, x@w1_i)@w2_i summed equals the single-device result."""
    r = _rng(7)
    x = r.standard_normal((2, 8))
    w1 = r.standard_normal((8, 32))
    w2 = r.standard_normal((32, 8))
    tp = 2
    sub = 32 // tp
    out_tp = sum(np.maximum(0.0, x @ w1[:, i * sub:(i + 1) * sub]) @ w2[i * sub:(i + 1) * sub, :]
                 for i in range(tp))
    _, _, Z = orc.mlp_fwd(x, w1, None, w2, None, act=_o.ACT_RELU)
    assert np.max(np.abs(Z - out_tp)) <= 1e-12 * np.max(np.abs(out_tp))


# --------------------------------------------------------------------------
# Backward ([M2] M025 追问: dW_i = X^T dY_i local, dX contributions summed;
#           M026: row-parallel dX_i = dY W_i^T is the input shard gradient;
#           M030: finite differences / gradcheck in double precision)

def _loss(orc, X, A, b1, B, b2, dZ, act):
    _, _, Z = orc.mlp_fwd(X, A, b1, B, b2, act=act)
    return float(np.sum(Z * dZ))


def pin_gradients_finite_difference(orc, act=_o.ACT_GELU):
    M, h, f = 4, 8, 32
    X, A, b1, B, b2, dZ = _problem(4, M, h, f, wscale=0.5)
    H, Y, _ = orc.mlp_fwd(X, A, b1, B, b2, act=act)
    g = orc.mlp_bwd(X, A, B, H, Y, dZ, act=act)
    params = {"X": X, "A": A, "B": B, "b1": b1, "b2": b2}
    names = {"X": "dX", "A": "dA", "B": "dB", "b1": "db1", "b2": "db2"}
    for name, arr in params.items():
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = arr[idx]
            eps = 1e-6 * max(1.0, abs(x0))
            arr[idx] = x0 + eps
            lp = _loss(orc, X, A, b1, B, b2, dZ, act)
            arr[idx] = x0 - eps
            lm = _loss(orc, X, A, b1, B, b2, dZ, act)
            arr[idx] = x0
            fd[idx] = (lp - lm) / (2 * eps)
        an = g[names[name]]
        err = np.linalg.norm(an - fd) / np.linalg.norm(fd)
        assert err <= 1e-6, (name, err)


def pin_identity_activation_backward_closed_form(orc):
    M, h, f = 7, 10, 15
    X, A, b1, B, b2, dZ = _problem(5, M, h, f)
    H, Y, _ = orc.mlp_fwd(X, A, b1, B, b2, act=_o.ACT_NONE)
    g = orc.mlp_bwd(X, A, B, H, Y, dZ, act=_o.ACT_NONE)
    dY = dZ @ B.T
    ref = {"dX": dY @ A.T, "dA": X.T @ dY, "dB": (X @ A + b1).T @ dZ,
           "db1": dY.sum(axis=0), "db2": dZ.sum(axis=0)}
    for k, v in ref.items():
        assert np.max(np.abs(g[k] - v)) <= 1e-12 * np.max(np.abs(v)), k


def pin_sharded_backward_equals_unsharded(orc):
    """Per shard: dA_i, dB_i, db1_i are the column / row slices of the unsharded
    gradients, and dX is the SUM of the shard contributions ([M2] M025 追问)."""
    M, h, f = 5, 6, 24
    X, A, b1, B, b2, dZ = _problem(6, M, h, f)
    H, Y, _ = orc.mlp_fwd(X, A, b1, B, b2)
    g = orc.mlp_bwd(X, A, B, H, Y, dZ)
    for p in (2, 3, 4, 6):
        fs = f // p
        dX_sum = np.zeros((M, h))
        for i in range(p):
            sl = slice(i * fs, (i + 1) * fs)
            Ai, Bi = np.ascontiguousarray(A[:, sl]), np.ascontiguousarray(B[sl, :])
            Hi, Yi, _ = orc.mlp_fwd(X, Ai, b1[sl], Bi, None)
            gi = orc.mlp_bwd(X, Ai, Bi, Hi, Yi, dZ)
            assert np.max(np.abs(gi["dA"] - g["dA"][:, sl])) <= 1e-12 * np.max(np.abs(g["dA"]))
            assert np.max(np.abs(gi["dB"] - g["dB"][sl, :])) <= 1e-12 * np.max(np.abs(g["dB"]))
            assert np.max(np.abs(gi["db1"] - g["db1"][sl])) <= 1e-12 * np.max(np.abs(g["db1"]))
            dX_sum += gi["dX"]
        assert np.max(np.abs(dX_sum - g["dX"])) <= 1e-12 * np.max(np.abs(g["dX"]))


def pin_sampled_backward_matches_full(orc):
    """The element-by-element sampled gradients agree with the (pinned) full backward."""
    M, h, f = 9, 8, 20
    X, A, b1, B, b2, dZ = _problem(8, M, h, f)
    H, Y, _ = orc.mlp_fwd(X, A, b1, B, b2)
    g = orc.mlp_bwd(X, A, B, H, Y, dZ)
    rows = [0, 3, 8]
    dXr = orc.bwd_dX_rows(X, A, b1, B, dZ, rows)
    assert np.max(np.abs(dXr - g["dX"][rows])) <= 1e-12 * np.max(np.abs(g["dX"]))
    cols = [0, 7, 19, 11]
    dAc, dBr, db1c = orc.bwd_ffn_cols(X, A, b1, B, dZ, cols)
    assert np.max(np.abs(dAc - g["dA"][:, cols])) <= 1e-12 * np.max(np.abs(g["dA"]))
    assert np.max(np.abs(dBr - g["dB"][cols, :])) <= 1e-12 * np.max(np.abs(g["dB"]))
    assert np.max(np.abs(db1c - g["db1"][cols])) <= 1e-12 * np.max(np.abs(g["db1"]))
    assert np.max(np.abs(orc.bwd_db2(dZ) - g["db2"])) <= 1e-12 * np.max(np.abs(g["db2"]))


# --------------------------------------------------------------------------
# Layout maps ([CP] 切分原理 / Python 演示 np.split; QKV interleave by heads)

def pin_shard_columns_vs_np_split(orc):
    r = _rng(9)
    for (rows, cols, p) in [(3, 12, 3), (5, 16, 4), (2, 8, 1), (4, 30, 5)]:
        W = r.integers(0, 2**16, size=(rows, cols), dtype=np.uint16)
        ref = np.stack(np.split(W, p, axis=1))
        assert np.array_equal(orc.shard_columns(W, p), ref)
        W32 = r.integers(0, 2**32, size=(rows, cols), dtype=np.uint32)
        assert np.array_equal(orc.shard_columns(W32, p), np.stack(np.split(W32, p, axis=1)))


def pin_qkv_interleave_heads_on_one_rank(orc):
    """Brute force: after the interleave, a p-way column split gives rank r exactly the
    Q, K and V columns of heads r*n/p .. (r+1)*n/p-1, in head order; and the map is a
    bijection whose inverse and adjoint are the transposed permutation."""
    for (h, n, p) in [(12, 4, 2), (24, 6, 3), (16, 8, 8), (8, 1, 1), (20, 5, 5)]:
        d = h // n
        rows = 3
        # label every source column by (t, head, e)
        src = np.empty((rows, 3 * h), dtype=np.int64)
        for t in range(3):
            for g in range(n):
                for e in range(d):
                    src[:, t * h + g * d + e] = 1_000_000 * t + 1000 * g + e
        dst = orc.qkv_interleave(src, h, n)
        cw = 3 * h // p
        hp = n // p
        for rk in range(p):
            block = dst[0, rk * cw:(rk + 1) * cw]
            expect = []
            for g in range(rk * hp, (rk + 1) * hp):
                for t in range(3):
                    expect += [1_000_000 * t + 1000 * g + e for e in range(d)]
            assert list(block) == expect
        # bijection + inverse
        perm = [orc.qkv_src_col(c, h, n) for c in range(3 * h)]
        assert sorted(perm) == list(range(3 * h))
        r = _rng(h + n)
        Wf = r.standard_normal((rows, 3 * h))
        assert np.array_equal(orc.qkv_interleave(orc.qkv_interleave(Wf, h, n), h, n, inverse=True), Wf)
        # adjoint: <S x, y> == <x, S^T y>
        Yf = r.standard_normal((rows, 3 * h))
        lhs = np.sum(orc.qkv_interleave(Wf, h, n) * Yf)
        rhs = np.sum(Wf * orc.qkv_interleave(Yf, h, n, inverse=True))
        assert abs(lhs - rhs) <= 1e-12 * abs(lhs) + 1e-12


# --------------------------------------------------------------------------
# Linear layer (attention projections; [M2] M025/M026, [TI] QKV by heads)

def pin_linear_vs_numpy_and_fd(orc):
    r = _rng(11)
    M, K, N = 7, 9, 12
    X = r.standard_normal((M, K)); W = r.standard_normal((K, N)); b = r.standard_normal(N)
    dY = r.standard_normal((M, N))
    Y = orc.linear_fwd(X, W, b)
    assert np.max(np.abs(Y - (X @ W + b))) <= 1e-13 * np.max(np.abs(Y))
    dX, dW, db = orc.linear_bwd(X, W, dY)
    for name, arr, g in (("X", X, dX), ("W", W, dW), ("b", b, db)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = arr[idx]
            eps = 1e-6 * max(1.0, abs(x0))
            arr[idx] = x0 + eps
            lp = float(np.sum(orc.linear_fwd(X, W, b) * dY))
            arr[idx] = x0 - eps
            lm = float(np.sum(orc.linear_fwd(X, W, b) * dY))
            arr[idx] = x0
            fd[idx] = (lp - lm) / (2 * eps)
        assert np.linalg.norm(g - fd) / np.linalg.norm(fd) <= 1e-7, name


def pin_qkv_interleave_commutes_with_projection(orc):
    """Permuting the projection's output columns equals projecting with the permuted
    weight (bit for bit: every output column is the same dot product), and the p-way
    column split of the interleaved projection gives each rank exactly its heads' q, k, v."""
    r = _rng(12)
    h, n, p, M = 24, 6, 3, 5
    X = r.standard_normal((M, h)); W = r.standard_normal((h, 3 * h)); b = r.standard_normal(3 * h)
    Y = orc.linear_fwd(X, W, b)
    Wi = orc.qkv_interleave(W, h, n)
    bi = orc.qkv_interleave(b.reshape(1, -1), h, n).reshape(-1)
    Yi = orc.linear_fwd(X, Wi, bi)
    assert np.array_equal(Yi, orc.qkv_interleave(Y, h, n))
    d, cw = h // n, 3 * h // p
    for rk in range(p):
        for g_local in range(n // p):
            g = rk * (n // p) + g_local
            for t in range(3):
                got = Yi[:, rk * cw + (3 * g_local + t) * d: rk * cw + (3 * g_local + t + 1) * d]
                assert np.array_equal(got, Y[:, t * h + g * d: t * h + (g + 1) * d])


# --------------------------------------------------------------------------
# SwiGLU variant ([M2] M027: gated activations work on local pairs of the shard)

def pin_silu_vs_library(orc):
    for x in np.linspace(-30.0, 30.0, 241):
        ref = x * special.expit(x)
        assert abs(orc.silu(x) - ref) <= 1e-15 * max(1.0, abs(ref)) + 1e-300
        eps = 1e-5
        fd = (orc.silu(x + eps) - orc.silu(x - eps)) / (2 * eps)
        assert abs(orc.silu_grad(x) - fd) < 1e-8
    assert orc.silu(0.0) == 0.0 and abs(orc.silu_grad(0.0) - 0.5) < 1e-16


def pin_swiglu_special_cases(orc):
    """U = 0, bu = 1: Y = silu(X G + bg), so Z = silu(H) B with scipy's expit; and G = 0 with a large
    gate bias (silu(40) = 40 up to 4e-17): the block is the affine map 40 (X U + bu) B + b2."""
    r = _rng(13)
    M, h, f = 6, 8, 20
    X = r.standard_normal((M, h)); G = r.standard_normal((h, f)) * 0.4; U = r.standard_normal((h, f)) * 0.4
    B = r.standard_normal((f, h)) * 0.4; bg = r.standard_normal(f) * 0.1; b2 = r.standard_normal(h) * 0.1
    Hg, _, _, Z = orc.swiglu_fwd(X, G, np.zeros((h, f)), bg, np.ones(f), B, b2)
    ref = (Hg * special.expit(Hg)) @ B + b2
    assert np.max(np.abs(Hg - (X @ G + bg))) <= 1e-13 * np.max(np.abs(Hg))
    assert np.max(np.abs(Z - ref)) <= 1e-13 * np.max(np.abs(ref))
    bu = r.standard_normal(f) * 0.1
    _, _, _, Z2 = orc.swiglu_fwd(X, np.zeros((h, f)), U, np.full(f, 40.0), bu, B, b2)
    ref2 = 40.0 * (X @ U + bu) @ B + b2
    assert np.max(np.abs(Z2 - ref2)) <= 1e-12 * np.max(np.abs(ref2))


def pin_swiglu_sharded_equals_unsharded(orc):
    """sum_i [silu(X G_i + bg_i) * (X U_i + bu_i)] B_i + b2 == the unsharded block, every divisor p."""
    r = _rng(14)
    M, h, f = 5, 6, 24
    X = r.standard_normal((M, h)); G = r.standard_normal((h, f)) * 0.4; U = r.standard_normal((h, f)) * 0.4
    B = r.standard_normal((f, h)) * 0.4; bg = r.standard_normal(f) * 0.1; bu = r.standard_normal(f) * 0.1
    b2 = r.standard_normal(h) * 0.1
    _, _, _, Z = orc.swiglu_fwd(X, G, U, bg, bu, B, b2)
    for p in _divisors(f):
        fs = f // p
        acc = np.zeros((M, h))
        for i in range(p):
            sl = slice(i * fs, (i + 1) * fs)
            _, _, _, Zi = orc.swiglu_fwd(X, np.ascontiguousarray(G[:, sl]), np.ascontiguousarray(U[:, sl]),
                                         bg[sl], bu[sl], np.ascontiguousarray(B[sl, :]), None)
            acc += Zi
        assert np.max(np.abs(acc + b2 - Z)) <= 1e-12 * np.max(np.abs(Z))


def pin_swiglu_gradients_finite_difference(orc):
    r = _rng(15)
    M, h, f = 3, 5, 8
    X = r.standard_normal((M, h)); G = r.standard_normal((h, f)) * 0.5; U = r.standard_normal((h, f)) * 0.5
    B = r.standard_normal((f, h)) * 0.5; bg = r.standard_normal(f) * 0.2; bu = r.standard_normal(f) * 0.2
    b2 = r.standard_normal(h) * 0.2; dZ = r.standard_normal((M, h))
    Hg, Hu, Y, _ = orc.swiglu_fwd(X, G, U, bg, bu, B, b2)
    g = orc.swiglu_bwd(X, G, U, B, Hg, Hu, Y, dZ)
    params = {"dX": X, "dG": G, "dU": U, "dB": B, "dbg": bg, "dbu": bu, "db2": b2}
    for name, arr in params.items():
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = arr[idx]
            eps = 1e-6 * max(1.0, abs(x0))
            arr[idx] = x0 + eps
            lp = float(np.sum(orc.swiglu_fwd(X, G, U, bg, bu, B, b2)[3] * dZ))
            arr[idx] = x0 - eps
            lm = float(np.sum(orc.swiglu_fwd(X, G, U, bg, bu, B, b2)[3] * dZ))
            arr[idx] = x0
            fd[idx] = (lp - lm) / (2 * eps)
        assert np.linalg.norm(g[name] - fd) / np.linalg.norm(fd) <= 1e-6, name


def pin_swiglu_pack_layout(orc):
    """Brute force: packed column 256 b + j of shard i holds gate (j < 128) or up feature
    i fs + 128 b + j mod 128; unpack inverts pack bit for bit."""
    rows, p, fs = 3, 2, 256
    f = p * fs
    G = np.arange(rows * f, dtype=np.int64).reshape(rows, f) * 2
    U = G + 1
    W = orc.swiglu_pack(G, U, p)
    for i in range(p):
        for c in range(2 * fs):
            b_, j = divmod(c, 256)
            src = G if j < 128 else U
            assert np.array_equal(W[i, :, c], src[:, i * fs + 128 * b_ + (j % 128)])
    G2, U2 = orc.swiglu_unpack(W, p)
    assert np.array_equal(G2, G) and np.array_equal(U2, U)


ALL_PINS = [
    pin_gelu_closed_forms,
    pin_gelu_vs_library,
    pin_column_concatenation_bitexact,
    pin_column_vs_numpy_demo,
    pin_row_sum_equals_unsharded,
    pin_identity_activation_vs_numpy,
    pin_relu_demo_structure,
    pin_gradients_finite_difference,
    pin_identity_activation_backward_closed_form,
    pin_sharded_backward_equals_unsharded,
    pin_sampled_backward_matches_full,
    pin_shard_columns_vs_np_split,
    pin_qkv_interleave_heads_on_one_rank,
    pin_linear_vs_numpy_and_fd,
    pin_qkv_interleave_commutes_with_projection,
    pin_silu_vs_library,
    pin_swiglu_special_cases,
    pin_swiglu_sharded_equals_unsharded,
    pin_swiglu_gradients_finite_difference,
    pin_swiglu_pack_layout,
]


def failing_pins(orc):
    """Names of the pins that fail (or crash) on this oracle build."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception:  # noqa: BLE001 - any failure counts
            bad.append(pin.__name__)
    return bad
