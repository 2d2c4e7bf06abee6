"""Sharding the GEMM + Amax over ranks, one process per GPU.

The C tiles are independent, so the work partitions with no data-path
exchange: every rank runs the single-GPU library on its own piece of the
problem, and the one collective is the max of the per-rank Amax values (a
4-byte all-reduce).  The pieces ("GEMM + Amax (SM100)", section "Shapes":
batched (M, K, L) x (N, K, L)):

* L >= world: whole batches, as evenly as possible;
* L == 1: M in whole 128-row scale atoms, so that every rank's SFA is a
  contiguous run of atoms and its A rows are contiguous;
* 1 < L < world: every rank takes one batch, and the ranks that share a
  batch split its M in whole atoms.

A rank's piece is a contiguous view of each tensor in the layouts the
library takes, so no copy is made.  An M split needs k-major A and n-major
C (an m-major operand or C would make the rank's rows a strided view); the
batch split works for every layout.  A rank may receive an empty piece (more
ranks than 128-row atoms): it launches nothing and contributes 0 to Amax.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class Shard:
    """Batches [l0, l1) and rows [m0, m1) of C owned by one rank."""
    l0: int
    l1: int
    m0: int
    m1: int

    @property
    def empty(self) -> bool:
        return self.l1 <= self.l0 or self.m1 <= self.m0

    @property
    def batches(self) -> int:
        return max(0, self.l1 - self.l0)

    @property
    def rows(self) -> int:
        return max(0, self.m1 - self.m0)


ATOM_ROWS = 128  # rows of one scale atom


def _split(n: int, parts: int, index: int) -> tuple[int, int]:
    """Part `index` of `parts` near-equal contiguous parts of range(n)."""
    return n * index // parts, n * (index + 1) // parts


def shard_of(M: int, L: int, world: int, rank: int) -> Shard:
    """The piece of an (M, N, L) problem that rank `rank` of `world` computes."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if M < 1 or L < 1:
        raise ValueError("empty problem")
    if L >= world:
        l0, l1 = _split(L, world, rank)
        return Shard(l0, l1, 0, M)
    # one batch per rank; the ranks on a batch split its rows in whole atoms
    l = rank * L // world
    first = -(-l * world // L)              # first rank on batch l
    last = -(-(l + 1) * world // L)         # one past its last rank
    atoms = -(-M // ATOM_ROWS)
    a0, a1 = _split(atoms, last - first, rank - first)
    return Shard(l, l + 1, min(M, a0 * ATOM_ROWS), min(M, a1 * ATOM_ROWS))


def local_problem(problem, shard: Shard):
    """A rank's problem: `problem` (a bsg_problem, or any dataclass with M
    and L fields) with the piece's rows and batches."""
    if shard.empty:
        raise ValueError("an empty shard has no problem")
    if dataclasses.is_dataclass(problem):
        return dataclasses.replace(problem, M=shard.rows, L=shard.batches)
    out = type(problem).from_buffer_copy(problem)
    out.M, out.L = shard.rows, shard.batches
    return out


def local_views(shard: Shard, A, B, SFA, SFB, C, *, M: int, a_major: str = "k",
                c_major: str = "n"):
    """Views of a rank's piece of the full tensors (torch tensors or numpy
    arrays in the library's layouts): A (L, M, Kb) or (L, K, M), B, the scale
    atom tensors (L, T, T_k, 32, 4, 4) and C (L, M, N[/2]) or (L, N, M).
    Whole-batch pieces slice the batch axis of everything; row pieces slice
    A, SFA and C inside one batch (k-major A and n-major C only)."""
    if shard.empty:
        raise ValueError("an empty shard has no tensors")
    bl = slice(shard.l0, shard.l1)
    if shard.rows == M:
        return A[bl], B[bl], SFA[bl], SFB[bl], C[bl]
    if a_major != "k" or c_major != "n":
        raise ValueError("a row split needs k-major A and n-major C")
    if shard.m0 % ATOM_ROWS:
        raise ValueError("a row split starts on a 128-row scale atom")
    rows = slice(shard.m0, shard.m1)
    atoms = slice(shard.m0 // ATOM_ROWS, -(-shard.m1 // ATOM_ROWS))
    return A[bl, rows], B[bl], SFA[bl, atoms], SFB[bl], C[bl, rows]


def allreduce_amax(amax, group=None) -> None:
    """Max of a one-element fp32 Amax tensor over the ranks, in place.  The
    reduction runs on the float's bit pattern as int32, the same integer max
    the kernel takes (Amax is non-negative; a NaN's bits order above every
    finite value, so a NaN on any rank wins)."""
    import torch
    import torch.distributed as dist
    bits = amax.view(torch.int32)
    dist.all_reduce(bits, op=dist.ReduceOp.MAX, group=group)
