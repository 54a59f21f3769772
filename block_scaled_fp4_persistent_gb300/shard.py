"""Splitting one grouped call across ranks (one GPU each), host side only.

A grouped call's outputs are independent: C_i[m][n] depends on row m of A_i and
row n of B_i alone, and no sum runs across groups or across n. So one call
shards with no exchange on the data path. Two plans:

 * by whole groups: each rank runs the groups assigned to it, whole. Groups go
   longest first, each to the rank with the least work so far; work is a
   group's algorithmic bytes (the call is HBM-bound), A, B, scales and C.
 * by N ranges: each rank runs every group, restricted to a contiguous range of
   B's rows (C's columns). Ranges are cut at multiples of 128 rows, so a range
   of prepacked scales is whole 128-row blocks, and are as equal as that allows.
   Each rank writes its column block of the group's C through ldc.

Either way C stays sharded: each rank holds (or writes into a shared buffer)
only its own outputs. An all-gather is up to the caller.

`sub_problem` restricts an Nvfp4Problem (of the C ABI) to a range of B's rows by
pointer arithmetic on its fields: B, SFB and C move, M, K and A stay. Nothing
here touches a GPU.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

ROW_ALIGN = 128  # N-range cuts fall on multiples of 128 rows (whole prepacked scale blocks)


def group_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one group: packed A and B, their scales, fp16 C."""
    return M * K // 2 + N * K // 2 + M * K // 16 + N * K // 16 + 2 * M * N


def shard_groups(shapes: Sequence[Tuple[int, int, int]], world: int) -> List[List[int]]:
    """Whole groups per rank: shapes is a list of (M, N, K); returns, for each rank,
    the indices of its groups in call order. Longest first to the least loaded rank
    (ties to the lowest rank), so every group lands on exactly one rank."""
    if world < 1:
        raise ValueError("world must be >= 1")
    load = [0] * world
    owner = [0] * len(shapes)
    order = sorted(range(len(shapes)), key=lambda i: -group_bytes(*shapes[i]))
    for i in order:
        r = min(range(world), key=lambda q: (load[q], q))
        owner[i] = r
        load[r] += group_bytes(*shapes[i])
    return [[i for i in range(len(shapes)) if owner[i] == r] for r in range(world)]


def n_ranges(N: int, world: int, align: int = ROW_ALIGN) -> List[Tuple[int, int]]:
    """Contiguous ranges [n0, n1) of 0..N, one per rank: cut r sits at the multiple of
    `align` nearest to r * N / world, so range sizes differ by at most `align`. A rank may
    get an empty range when N has fewer aligned blocks than ranks."""
    if world < 1:
        raise ValueError("world must be >= 1")
    cuts = [0]
    for r in range(1, world):
        c = min(N, (r * N + world * align // 2) // (world * align) * align)
        cuts.append(max(c, cuts[-1]))
    cuts.append(N)
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def shard_n(shapes: Sequence[Tuple[int, int, int]], world: int) -> List[List[Tuple[int, int, int]]]:
    """N ranges per rank: for each rank, a list of (group, n0, n1) with n1 > n0, every
    group's columns covered exactly once over all ranks."""
    per = [[] for _ in range(world)]
    for g, (M, N, K) in enumerate(shapes):
        for r, (n0, n1) in enumerate(n_ranges(N, world)):
            if n1 > n0:
                per[r].append((g, n0, n1))
    return per


def prepacked_row_offset(rows: int, K: int) -> int:
    """Bytes of the blocked scale layout before row `rows` (a multiple of 128)."""
    if rows % ROW_ALIGN:
        raise ValueError("prepacked scales can only be cut at multiples of 128 rows")
    return (rows // 128) * ((K + 63) // 64) * 512


def sub_problem(p, n0: int, n1: int, problem_type):
    """The problem restricted to B's rows n0..n1-1 (C's columns), as a new
    `problem_type` (the binding's Nvfp4Problem). B, SFB and C move; C keeps the
    parent's row stride through ldc. n0 must be a multiple of 128 unless n0 == 0."""
    from . import NVFP4_SF_PREPACKED  # the binding's constants
    if not (0 <= n0 < n1 <= p.N):
        raise ValueError(f"bad range {n0}..{n1} of N = {p.N}")
    if n0 % ROW_ALIGN:
        raise ValueError("N ranges start at multiples of 128")
    K = p.K
    ldc = p.ldc if p.ldc else p.N
    if p.sf_layout == NVFP4_SF_PREPACKED:
        sfb = p.SFB + prepacked_row_offset(n0, K)
    else:
        sfb = p.SFB + n0 * (K // 16)
    return problem_type(p.M, n1 - n0, K, p.sf_layout, p.A, p.B + n0 * (K // 2), p.SFA, sfb, p.C + 2 * n0, ldc, 0)


def rank_problems(probs, world: int, rank: int, mode: str):
    """This rank's share of one grouped call: the problems it runs, in call order.
    mode 'groups' (whole groups) or 'n' (N ranges of every group)."""
    shapes = [(p.M, p.N, p.K) for p in probs]
    if mode == "groups":
        return [probs[i] for i in shard_groups(shapes, world)[rank]]
    if mode == "n":
        ptype = type(probs[0]) if probs else None
        return [sub_problem(probs[g], n0, n1, ptype) for g, n0, n1 in shard_n(shapes, world)[rank]]
    raise ValueError(f"unknown shard mode {mode!r}")
