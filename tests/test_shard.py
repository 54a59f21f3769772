"""Splitting one grouped call across ranks, on CPU.

The plans of `block_scaled_fp4_persistent_gb300.shard` (whole groups, N ranges) are
checked for coverage and balance, `sub_problem` for its pointer arithmetic, and two gloo
ranks each compute their share of one call with the oracle: the union of their outputs
covers every output exactly once and equals the single-process oracle's result bit for
bit. (On GPUs each rank runs its share through the C ABI, writing its column block of C
through ldc; `tests/test_shard_gpu.py` runs the shares one after another on one GPU.)
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import gen
from block_scaled_fp4_persistent_gb300 import shard
import block_scaled_fp4_persistent_gb300 as nv

SHAPES = [(40, 384, 512), (200, 520, 256), (130, 256, 768), (7, 8, 64), (64, 1024, 256)]


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_whole_groups_cover_every_group_once_and_balance(world):
    plan = shard.shard_groups(SHAPES, world)
    assert sorted(i for r in plan for i in r) == list(range(len(SHAPES)))
    assert all(r == sorted(r) for r in plan)
    load = [sum(shard.group_bytes(*SHAPES[i]) for i in r) for r in plan]
    biggest = max(shard.group_bytes(*s) for s in SHAPES)
    assert max(load) - min(load) <= biggest


@pytest.mark.parametrize("N,world", [(520, 2), (4096, 8), (128, 3), (8, 2), (7168, 3), (136, 2)])
def test_n_ranges_are_aligned_contiguous_and_cover(N, world):
    r = shard.n_ranges(N, world)
    assert len(r) == world and r[0][0] == 0 and r[-1][1] == N
    for (a0, a1), (b0, _) in zip(r, r[1:]):
        assert a1 == b0 and a0 <= a1
    assert all(n0 % 128 == 0 for n0, _ in r)
    sizes = [n1 - n0 for n0, n1 in r]
    assert max(sizes) - min(sizes) <= 128


def test_shard_n_covers_every_column_once():
    plan = shard.shard_n(SHAPES, 3)
    for g, (M, N, K) in enumerate(SHAPES):
        cols = np.zeros(N, int)
        for r in plan:
            for gg, n0, n1 in r:
                if gg == g:
                    cols[n0:n1] += 1
        assert (cols == 1).all()


def test_sub_problem_moves_b_sfb_and_c():
    M, N, K = 40, 520, 512
    base = dict(A=0x10000, B=0x20000, SFA=0x30000, SFB=0x40000, C=0x50000)
    for layout in (nv.NVFP4_SF_PREPACKED, nv.NVFP4_SF_ROWMAJOR):
        p = nv.Nvfp4Problem(M, N, K, layout, base["A"], base["B"], base["SFA"], base["SFB"], base["C"], 0, 0)
        q = shard.sub_problem(p, 256, 520, nv.Nvfp4Problem)
        assert (q.M, q.N, q.K, q.sf_layout, q.ldc) == (M, 264, K, layout, N)
        assert q.A == base["A"] and q.SFA == base["SFA"]
        assert q.B == base["B"] + 256 * K // 2
        assert q.C == base["C"] + 2 * 256
        step = 2 * 8 * 512 if layout == nv.NVFP4_SF_PREPACKED else 256 * K // 16  # 2 blocks of 128 rows x 8 atoms
        assert q.SFB == base["SFB"] + step
    with pytest.raises(ValueError):
        shard.sub_problem(p, 100, 200, nv.Nvfp4Problem)  # not a multiple of 128


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _groups():
    Ms, Ns, Ks = zip(*SHAPES)
    return gen.make_problem_set(91, list(Ms), list(Ns), list(Ks))


def _rank_main(rank, world, port, mode, out):
    import torch
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    groups = _groups()
    flat = sum(g.M * g.N for g in groups)
    offs = np.cumsum([0] + [g.M * g.N for g in groups])
    c_bits = torch.zeros(flat, dtype=torch.int32)
    cover = torch.zeros(flat, dtype=torch.int32)
    shapes = [(g.M, g.N, g.K) for g in groups]
    if mode == "groups":
        mine = [(i, 0, groups[i].N) for i in shard.shard_groups(shapes, world)[rank]]
    else:
        mine = shard.shard_n(shapes, world)[rank]
    for gi, n0, n1 in mine:
        g = groups[gi]
        sub = gen.GroupInputs(g.M, n1 - n0, g.K, g.A, g.B[n0:n1], g.SFA, g.SFB[n0:n1])
        (c, _), = oracle.grouped_gemm([sub])
        block = np.zeros((g.M, g.N), np.int32)
        hit = np.zeros((g.M, g.N), np.int32)
        block[:, n0:n1] = c.view(np.uint16).astype(np.int32)
        hit[:, n0:n1] = 1
        c_bits[offs[gi]:offs[gi + 1]] += torch.from_numpy(block.reshape(-1))
        cover[offs[gi]:offs[gi + 1]] += torch.from_numpy(hit.reshape(-1))
    dist.all_reduce(c_bits)
    dist.all_reduce(cover)
    if rank == 0:
        out["bits"] = c_bits.numpy().copy()
        out["cover"] = cover.numpy().copy()
    dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["groups", "n"])
def test_two_gloo_ranks_compute_one_call_exactly_once(mode):
    import oracle
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), mode, out), nprocs=world, start_method="spawn",
                       join=True)
    assert (out["cover"] == 1).all(), "an output computed by no rank or by two"
    ref = np.concatenate([c.view(np.uint16).astype(np.int32).reshape(-1) for c, _ in oracle.grouped_gemm(_groups())])
    assert np.array_equal(out["bits"], ref)
