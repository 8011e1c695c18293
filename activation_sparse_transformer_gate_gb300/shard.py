"""Token-sharded data parallelism for the sparse FFN's training step.

The FFN is per-token: the forward (gate GEMM, TwELL pack, hybrid split, up /
down projections) and the backward's dh and dx need nothing from other
tokens, so a batch of T tokens splits into contiguous token ranges, one per
rank, with no exchange on the forward or for dx.  The weight gradients
dW_gate, dW_up, dW_down and dbg are sums over tokens: each rank's backward
computes its range's partial sums (fp32), and one all-reduce (sum) over the
ranks gives the batch's gradients.  (Splitting the neurons instead -- whole
TwELL tiles per rank, which are independent by construction -- would need
one all-reduce of y and of dx instead.)

Host-side plumbing only: the ranges and the collective.  Every step of the
FFN runs in the library's kernels on each rank's device; the reduction is
torch.distributed's all_reduce (NCCL on GPUs, gloo on the CPU).
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple


def token_range(T: int, rank: int, world: int, align: int = 128) -> Tuple[int, int]:
    """[start, end) of the tokens of `rank` when T tokens are split over
    `world` ranks: contiguous ranges of whole blocks of `align` tokens (the
    tensor-core row tile), as even as whole blocks allow; the last range
    takes the ragged tail.  Ranges may be empty when T < world * align."""
    if T < 0 or world < 1 or not 0 <= rank < world or align < 1:
        raise ValueError(f"token_range: T={T} rank={rank} world={world} align={align}")
    blocks = (T + align - 1) // align
    base, extra = divmod(blocks, world)
    b0 = rank * base + min(rank, extra)
    b1 = b0 + base + (1 if rank < extra else 0)
    return min(T, b0 * align), min(T, b1 * align)


def allreduce_weight_grads(grads: Iterable, group: Optional[object] = None) -> None:
    """Sum each rank's partial weight gradients (dW_gate, dW_up, dW_down,
    dbg; fp32 tensors, None entries skipped) over the ranks, in place.
    Every rank must pass the same tensors in the same order."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        raise RuntimeError("allreduce_weight_grads needs an initialised process group")
    for g in grads:
        if g is not None:
            dist.all_reduce(g, op=dist.ReduceOp.SUM, group=group)
