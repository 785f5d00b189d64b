"""The block with its shards spread over the ranks of a tensor-parallel group (GPU).

Rank r computes its partial through tpmlp_mlp_fwd_partial / tpmlp_mlp_bwd_partial on its own
FFN features ("分布式并行训练全景", 考点 2; "Megatron 专家面试题 Level 2", M025 追问, M026), the
partials are summed (the All-Reduce), and tpmlp_sum_finish adds b2 once and rounds.

* Ranks emulated one after another on one GPU: each rank's kernels run on its slice of the
  weights, the fp32 partials are summed in rank order (standing in for the All-Reduce; no
  kernel waits on another), and the results are compared with the fp64 oracle of the
  unsharded block.
* A one-rank NCCL group through the driver's real All-Reduce: with every shard on one rank the
  result is bit-identical to tpmlp_mlp_fwd / tpmlp_mlp_bwd (same kernels, same accumulation
  order; the finish step rounds the same fp32 value).
* Two ranks on two GPUs with NCCL: skipped when fewer than two GPUs are visible.
"""
import os
import socket
import sys

import numpy as np
import pytest

import gpu_util as U

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth, tp
    from megatron_tensor_mlp_gb300 import tpmlp as T
    return harness, synth, tp, T


def _rank_weights(harness, T, buf, lo, hi, p_local):
    """Rank weights in the shard layout: A's columns, b1's entries, B's rows [lo, hi)."""
    import torch
    host = buf.host
    h, fr = buf.wl.h, hi - lo
    A = harness.to_torch(np.ascontiguousarray(host["A"][:, lo:hi]))
    A_sh = torch.empty((p_local, h, fr // p_local), dtype=A.dtype, device="cuda")
    T.tpmlp_shard_columns(A, A_sh, h, fr, p_local, buf.dt)
    B_sh = harness.to_torch(np.ascontiguousarray(host["B"][lo:hi])).view(p_local, fr // p_local, h)
    b1 = None if host["b1"] is None else harness.to_torch(np.ascontiguousarray(host["b1"][lo:hi])).view(p_local, -1)
    return A_sh, b1, B_sh


@pytest.mark.parametrize("world,p_local", [(2, 1), (4, 1), (2, 2)])
def test_emulated_ranks_match_the_oracle(env, orc, world, p_local):
    import torch
    harness, synth, tp, T = env
    wl = synth.custom(100, 3, 264, 2112, world * p_local, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=61)
    buf = harness.MLPBuffers(wl, backward=True)
    s, b, h, f, _ = buf.dims()
    M = s * b
    Z_sum = torch.zeros((M, h), dtype=torch.float32, device="cuda")
    dX_sum = torch.zeros((M, h), dtype=torch.float32, device="cuda")
    grads = []
    for r in range(world):
        lo, hi = tp.feature_range(r, world, f)
        A_sh, b1, B_sh = _rank_weights(harness, T, buf, lo, hi, p_local)
        ops = tp.LibraryRankOps(s, b, h, hi - lo, p_local)
        Zp, Y, H = ops.fwd_partial(buf.X, A_sh, b1, B_sh)
        Z_sum += Zp  # the All-Reduce, in rank order
        g = ops.bwd_partial(buf.X, A_sh, B_sh, H, Y, buf.dZ)
        dX_sum += g["dX_part"]
        grads.append({k: g[k].clone() for k in ("dA", "dB", "db1", "db2")})
    Z = ops.finish(Z_sum, buf.b2)
    dX = ops.finish(dX_sum, None)
    T.tpmlp_device_status()
    x = U.host_inputs_f64(buf)
    Hr, Yr, Zr = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    gr = orc.mlp_bwd(x["X"], x["A"], x["B"], Hr, Yr, x["dZ"])
    U.assert_close(harness.to_host(Z), Zr, "bf16", "Z")
    U.assert_close(harness.to_host(dX), gr["dX"], "bf16", "dX")
    dA = torch.cat([g["dA"].permute(1, 0, 2).reshape(h, -1) for g in grads], dim=1)
    dB = torch.cat([g["dB"].reshape(-1, h) for g in grads], dim=0)
    db1 = torch.cat([g["db1"].reshape(-1) for g in grads])
    U.assert_close(harness.to_host(dA), gr["dA"], "bf16", "dA")
    U.assert_close(harness.to_host(dB), gr["dB"], "bf16", "dB")
    U.assert_close(harness.to_host(db1), gr["db1"], "bf16", "db1")
    for g in grads:
        U.assert_close(harness.to_host(g["db2"]), gr["db2"], "bf16", "db2")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_one_rank_nccl_group_is_bit_identical(env):
    """The driver's real All-Reduce (NCCL, one rank): Z, dX and every gradient bit-identical to
    the single-GPU block."""
    import torch
    import torch.distributed as dist
    harness, synth, tp, T = env
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    wl = synth.custom(90, 4, 520, 2080, 2, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=62)
    buf = harness.MLPBuffers(wl, backward=True)
    s, b, h, f, p = buf.dims()
    buf.fwd()
    buf.bwd()
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    try:
        ops = tp.LibraryRankOps(s, b, h, f, p)
        ar = tp.process_group_all_reduce()
        Z, Y, H = tp.tp_mlp_fwd(ops, ar, buf.X, buf.A_sh, buf.b1_sh, buf.B_sh, buf.b2)
        g = tp.tp_mlp_bwd(ops, ar, buf.X, buf.A_sh, buf.B_sh, H, Y, buf.dZ)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    T.tpmlp_device_status()
    assert torch.equal(Z, buf.Z) and torch.equal(Y, buf.Y) and torch.equal(H, buf.H)
    assert torch.equal(g["dX"], buf.dX)
    for k, ref in (("dA", buf.dA_sh), ("dB", buf.dB_sh), ("db1", buf.db1_sh), ("db2", buf.db2)):
        assert torch.equal(g[k], ref), k


def _two_gpu_worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from megatron_tensor_mlp_gb300 import harness, synth, tp
    from megatron_tensor_mlp_gb300 import tpmlp as T
    torch.cuda.set_device(rank)
    dist.init_process_group("nccl", rank=rank, world_size=2)
    try:
        wl = synth.custom(64, 4, 256, 2048, 2, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=63)
        buf = harness.MLPBuffers(wl, backward=True)
        s, b, h, f, _ = buf.dims()
        lo, hi = tp.feature_range(rank, 2, f)
        A_sh, b1, B_sh = _rank_weights(harness, T, buf, lo, hi, 1)
        ops = tp.LibraryRankOps(s, b, h, hi - lo, 1)
        ar = tp.process_group_all_reduce()
        Z, Y, H = tp.tp_mlp_fwd(ops, ar, buf.X, A_sh, b1, B_sh, buf.b2)
        g = tp.tp_mlp_bwd(ops, ar, buf.X, A_sh, B_sh, H, Y, buf.dZ)
        torch.cuda.synchronize()
        q.put((rank, harness.to_host(Z), harness.to_host(g["dX"])))
    finally:
        dist.destroy_process_group()


def test_two_gpus_nccl(env, orc):
    import torch
    import torch.multiprocessing as mp
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    harness, synth, _, _ = env
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_two_gpu_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted([q.get(timeout=600) for _ in range(2)], key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    wl = synth.custom(64, 4, 256, 2048, 2, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=63)
    x = {k: synth.widen(wl.gen(k)) for k in ("X", "A", "B", "b1", "b2", "dZ")}
    H, Y, Z = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    g = orc.mlp_bwd(x["X"], x["A"], x["B"], H, Y, x["dZ"])
    for rank, Zr, dXr in out:
        U.assert_close(Zr, Z, "bf16", f"Z rank {rank}")
        U.assert_close(dXr, g["dX"], "bf16", f"dX rank {rank}")


@pytest.mark.parametrize("rows,cols,with_bias,dt", [(1, 8, True, 0), (37, 264, True, 0), (512, 1024, False, 0),
                                                  (37, 260, True, 1), (0, 64, True, 0)],
                         ids=["one-row", "ragged", "no-bias", "fp32", "empty"])
def test_sum_finish_bit_exact(env, rows, cols, with_bias, dt):
    """round(S + bias) once, after the All-Reduce: bit-exact against torch's own fp32 add and
    round-to-nearest-even conversion (bf16), or the plain fp32 sum."""
    import torch
    _, _, _, T = env
    g = torch.Generator(device="cuda").manual_seed(rows * 7 + cols)
    n = max(rows, 1)  # an empty call still passes valid buffers (pointers are checked first)
    S = torch.randn((n, cols), dtype=torch.float32, device="cuda", generator=g) * 3.0
    odt = torch.bfloat16 if dt == T.BF16 else torch.float32
    bias = (torch.randn((cols,), dtype=torch.float32, device="cuda", generator=g).to(odt)) if with_bias else None
    out = torch.full((n, cols), float("nan"), dtype=odt, device="cuda")
    T.tpmlp_sum_finish(S, bias, out, rows, cols, dt=dt)
    T.tpmlp_device_status()
    want = (S + (bias.float() if with_bias else 0.0)).to(odt)
    iv = torch.int16 if dt == T.BF16 else torch.int32
    assert torch.equal(out[:rows].view(iv), want[:rows].view(iv))
    if rows == 0:
        assert bool(torch.isnan(out.float()).all())  # nothing written


def test_emulated_ranks_fp32(env, orc):
    """The fp32 path of the rank-local entry points (FMA GEMMs, no TF32): two ranks emulated on
    one GPU, relative Frobenius error <= 1e-5 against the oracle."""
    import torch
    harness, synth, tp, T = env
    wl = synth.custom(8, 2, 64, 256, 2, dtype="f32", sigma_w=0.05, sigma_bias=0.05, seed=64)
    buf = harness.MLPBuffers(wl, backward=True)
    s, b, h, f, _ = buf.dims()
    M = s * b
    Z_sum = torch.zeros((M, h), dtype=torch.float32, device="cuda")
    dX_sum = torch.zeros((M, h), dtype=torch.float32, device="cuda")
    for r in range(2):
        lo, hi = tp.feature_range(r, 2, f)
        A_sh, b1, B_sh = _rank_weights(harness, T, buf, lo, hi, 1)
        ops = tp.LibraryRankOps(s, b, h, hi - lo, 1, dt=T.F32)
        Zp, Y, H = ops.fwd_partial(buf.X, A_sh, b1, B_sh)
        Z_sum += Zp
        dX_sum += ops.bwd_partial(buf.X, A_sh, B_sh, H, Y, buf.dZ)["dX_part"]
    Z, dX = ops.finish(Z_sum, buf.b2), ops.finish(dX_sum, None)
    T.tpmlp_device_status()
    x = U.host_inputs_f64(buf)
    Hr, Yr, Zr = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    gr = orc.mlp_bwd(x["X"], x["A"], x["B"], Hr, Yr, x["dZ"])
    U.assert_close(harness.to_host(Z), Zr, "f32", "Z")
    U.assert_close(harness.to_host(dX), gr["dX"], "f32", "dX")
