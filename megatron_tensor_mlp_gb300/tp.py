"""The MLP block with its shards spread over the GPUs of a tensor-parallel group.

Pages: "分布式并行训练全景", 考点 2 (each card holds a column slice of the first
weight and the matching row slice of the second and computes GeLU(X A_i) B_i; the
partial outputs are summed by one All-Reduce); "Megatron 专家面试题 Level 2",
M025 追问 (backward: weight gradients stay local, the dX contributions are summed
by an All-Reduce), M026 (row-parallel layer: the sum of the partials is the output)
and M027 (column -> GeLU -> row needs that one sum at the end of the block only).

Rank r of a group of `world` ranks owns FFN features [r ffn/world, (r+1) ffn/world):
those columns of A and b1 and those rows of B, held as p_local shards in the
library's shard layout.  A step is

    forward    Z_part = rank-local block (fp32, no b2)   tpmlp_mlp_fwd_partial
               all_reduce(Z_part)                         the caller's collective
               Z = round(Z_part + b2)                     tpmlp_sum_finish
    backward   dX_part, dA_r, dB_r, db1_r, db2            tpmlp_mlp_bwd_partial
               all_reduce(dX_part)
               dX = round(dX_part)                        tpmlp_sum_finish

The rank-local compute and the All-Reduce are parameters of the step functions,
so the same driver runs on GPUs (LibraryRankOps and NCCL) and in CPU tests (any
object with the same three methods, and gloo).  Nothing here computes any of the
block's arithmetic itself.
"""
from __future__ import annotations

from . import tpmlp as T


def feature_range(rank: int, world: int, ffn: int) -> tuple[int, int]:
    """FFN features [lo, hi) of A's columns, b1 and B's rows owned by `rank`."""
    if world < 1 or not 0 <= rank < world or ffn % world != 0:
        raise ValueError(f"ffn={ffn} must split evenly over {world} ranks (rank {rank})")
    n = ffn // world
    return rank * n, (rank + 1) * n


def tp_mlp_fwd(ops, all_reduce, X, A_sh, b1_sh, B_sh, b2):
    """Forward of the block on this rank: local partial, All-Reduce, b2 once.
    Returns (Z, Y, H); Y and H are this rank's shards, kept for the backward."""
    Z_part, Y, H = ops.fwd_partial(X, A_sh, b1_sh, B_sh)
    all_reduce(Z_part)
    return ops.finish(Z_part, b2), Y, H


def tp_mlp_bwd(ops, all_reduce, X, A_sh, B_sh, H, Y, dZ):
    """Backward on this rank: dict with dX (summed over the group) and the local dA, dB, db1,
    and db2 (the same on every rank)."""
    g = ops.bwd_partial(X, A_sh, B_sh, H, Y, dZ)
    all_reduce(g["dX_part"])
    g["dX"] = ops.finish(g["dX_part"], None)
    return g


def process_group_all_reduce(group=None):
    """In-place sum over a torch.distributed process group (NCCL between GPUs)."""
    import torch.distributed as dist

    def all_reduce(t):
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)

    return all_reduce


class LibraryRankOps:
    """Rank-local compute on this GPU through the C-ABI, with buffers allocated once (torch
    supplies the memory).  ffn_local and p_local are this rank's FFN width and shard count."""

    def __init__(self, s, b, h, ffn_local, p_local, dt=T.BF16, grad_dt=T.F32, stream=None, device="cuda"):
        import torch
        self.dims = (s, b, h, ffn_local, p_local)
        self.dt, self.grad_dt, self.stream = dt, grad_dt, stream
        M, fs = s * b, ffn_local // p_local
        tdt = torch.bfloat16 if dt == T.BF16 else torch.float32
        gdt = torch.float32 if grad_dt == T.F32 else torch.bfloat16
        e = lambda shape, d: torch.empty(shape, dtype=d, device=device)  # noqa: E731
        self.Y, self.H, self.dH = e((p_local, M, fs), tdt), e((p_local, M, fs), tdt), e((p_local, M, fs), tdt)
        self.Z_part, self.dX_part = e((M, h), torch.float32), e((M, h), torch.float32)
        self.Z, self.dX = e((M, h), tdt), e((M, h), tdt)
        self.dA, self.dB = e((p_local, h, fs), gdt), e((p_local, fs, h), gdt)
        self.db1, self.db2 = e((p_local, fs), gdt), e((h,), gdt)

    def fwd_partial(self, X, A_sh, b1_sh, B_sh):
        T.tpmlp_mlp_fwd_partial(X, A_sh, b1_sh, B_sh, self.Z_part, self.Y, self.H, *self.dims, dt=self.dt,
                                stream=self.stream)
        return self.Z_part, self.Y, self.H

    def bwd_partial(self, X, A_sh, B_sh, H, Y, dZ):
        T.tpmlp_mlp_bwd_partial(X, A_sh, B_sh, H, Y, dZ, self.dX_part, self.dA, self.dB, self.db1, self.db2,
                                self.dH, *self.dims, dt=self.dt, grad_dt=self.grad_dt, stream=self.stream)
        return {"dX_part": self.dX_part, "dA": self.dA, "dB": self.dB, "db1": self.db1, "db2": self.db2}

    def finish(self, S, bias):
        """round(S + bias) into Z (S = this rank's summed Z_part), dX (S = dX_part) or, for any
        other fp32 sum, a new tensor."""
        import torch
        if S is self.Z_part:
            out = self.Z
        elif S is self.dX_part:
            out = self.dX
        else:
            out = torch.empty(S.shape, dtype=self.Z.dtype, device=S.device)
        M, h = S.shape
        T.tpmlp_sum_finish(S, bias, out, M, h, dt=self.dt, stream=self.stream)
        return out
