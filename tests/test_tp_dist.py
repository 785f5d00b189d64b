"""The block split over several ranks, with the All-Reduce (CPU, gloo; no GPU).

"分布式并行训练全景", 考点 2 and "Megatron 专家面试题 Level 2", M025 追问 / M026 / M027: rank r
holds A's columns, b1's entries and B's rows of its FFN features, computes its partial
GeLU(X A_r + b1_r) B_r, and one All-Reduce sums the partials; b2 is added once, after the
sum.  In the backward dA_r, dB_r, db1_r stay local and the dX contributions are summed.

The driver (megatron_tensor_mlp_gb300.tp) runs here with gloo ranks and a rank-local
compute built on the oracle (each rank's partial is the oracle's block on that rank's
slice), so the test checks the driver's data flow against the unsharded oracle: every
rank's Z and dX within 1e-12 (fp64 reassociation), the local gradients equal to the
unsharded ones' slices.  A planted mistake (b2 added on every rank before the sum) must
fail the same comparison.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPE = (6, 3, 16, 64)  # s, b, h, ffn


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleRankOps:
    """Rank-local compute for the CPU test: the oracle's block on this rank's slice."""

    def __init__(self, orc, b2_per_rank=None):
        self.orc, self.b2_per_rank = orc, b2_per_rank

    def fwd_partial(self, X, A_r, b1_r, B_r):
        import torch
        H, Y, Zp = self.orc.mlp_fwd(X, A_r, b1_r, B_r, self.b2_per_rank)  # b2 only in the planted mistake
        return torch.from_numpy(Zp), Y, H

    def bwd_partial(self, X, A_r, B_r, H, Y, dZ):
        import torch
        g = self.orc.mlp_bwd(X, A_r, B_r, H, Y, dZ)
        return {"dX_part": torch.from_numpy(g["dX"]), "dA": g["dA"], "dB": g["dB"], "db1": g["db1"],
                "db2": g["db2"]}

    def finish(self, S, bias):
        out = S.numpy().copy()
        if bias is not None:
            out += bias
        return out


def _inputs(world):
    from megatron_tensor_mlp_gb300 import synth
    s, b, h, ffn = SHAPE
    wl = synth.custom(s, b, h, ffn, world, dtype="bf16", sigma_w=0.1, sigma_bias=0.1, seed=21)
    return {k: synth.widen(wl.gen(k)) for k in ("X", "A", "B", "b1", "b2", "dZ")}


def _worker(rank, world, port, q, mutant):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from megatron_tensor_mlp_gb300 import tp

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _inputs(world)
        lo, hi = tp.feature_range(rank, world, x["A"].shape[1])
        A_r, B_r, b1_r = x["A"][:, lo:hi], x["B"][lo:hi], x["b1"][lo:hi]
        ops = OracleRankOps(oracle.get(), b2_per_rank=x["b2"] if mutant else None)
        ar = tp.process_group_all_reduce()
        Z, Y, H = tp.tp_mlp_fwd(ops, ar, x["X"], A_r, b1_r, B_r, x["b2"])
        g = tp.tp_mlp_bwd(ops, ar, x["X"], A_r, B_r, H, Y, x["dZ"])
        q.put((rank, lo, hi, Z, g["dX"], g["dA"], g["dB"], g["db1"], g["db2"]))
    finally:
        dist.destroy_process_group()


def _run(world, mutant=False):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, mutant)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda t: t[0])


def _rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(b))


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_over_ranks_equals_unsharded(orc, world):
    x = _inputs(world)
    H, Y, Z = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    g = orc.mlp_bwd(x["X"], x["A"], x["B"], H, Y, x["dZ"])
    ranks = _run(world)
    dA = np.concatenate([r[5] for r in ranks], axis=1)
    dB = np.concatenate([r[6] for r in ranks], axis=0)
    db1 = np.concatenate([r[7] for r in ranks])
    for rank, lo, hi, Zr, dXr, dAr, dBr, db1r, db2r in ranks:
        assert _rel(Zr, Z) <= 1e-12, (rank, _rel(Zr, Z))       # summed partials + b2 once
        assert _rel(dXr, g["dX"]) <= 1e-12, rank                 # summed dX contributions
        assert _rel(db2r, g["db2"]) <= 1e-12, rank               # the same db2 on every rank
        assert (hi - lo) * world == x["A"].shape[1]
    assert _rel(dA, g["dA"]) <= 1e-12 and _rel(dB, g["dB"]) <= 1e-12 and _rel(db1, g["db1"]) <= 1e-12


def test_bias_added_on_every_rank_is_caught(orc):
    """Planted mistake: each rank adds b2 to its partial, so the sum carries (world + 1) b2."""
    world = 2
    x = _inputs(world)
    _, _, Z = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    ranks = _run(world, mutant=True)
    assert _rel(ranks[0][3], Z) > 1e-3


def test_feature_range_partitions_the_ffn_width():
    from megatron_tensor_mlp_gb300 import tp
    for world in (1, 2, 3, 4, 8):
        spans = [tp.feature_range(r, world, 96) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == 96
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    with pytest.raises(ValueError):
        tp.feature_range(0, 5, 96)
