"""C column blocks through ldc, and one grouped call run as several ranks' shares, on one GPU.

 * ldc: every kernel kind writes each group's C as a column block of a wider row-major
   matrix; every output is compared with the oracle and the columns around each block
   (filled with a canary) must stay untouched, K == 0 groups included.
 * shards: the shares that `block_scaled_fp4_persistent_gb300.shard` plans for 2 and 3
   ranks (whole groups, N ranges) run one after another, each through the C ABI, into one
   C; together they must produce every output of the call, within the acceptance bound.
   (Ranks on separate GPUs run the same calls, one each; nothing crosses between them.)
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity import assert_within_bound
import block_scaled_fp4_persistent_gb300 as nv
from block_scaled_fp4_persistent_gb300 import shard
from gpu_util import CANARY, DeviceGroup, workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    yield
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 0)


@pytest.mark.parametrize("kind", [0, 1, 2, 3, 4])
def test_column_blocks_through_ldc(kind):
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, kind)
    groups = gen.make_problem_set(401, [130, 40, 7, 64], [264, 512, 8, 136], [1024, 512, 64, 0])
    d = [DeviceGroup(g) for g in groups]
    M = max(g.M for g in groups)
    # one wide C: group i's block at columns off[i] .. off[i] + N_i, with 8 canary columns between
    off, w = [], 8
    for g in groups:
        off.append(w)
        w += g.N + 8
    wide = torch.full((M, w), CANARY, dtype=torch.int16, device="cuda").view(torch.float16)
    probs = []
    for i, (g, x) in enumerate(zip(groups, d)):
        p = x.problem()
        p.C = wide[:, off[i]:].data_ptr()
        p.ldc = w
        probs.append(p)
    nv.nvfp4_grouped_gemm(probs)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status()[0] == 0
    got = wide.cpu().numpy()
    mask = np.ones(got.shape, bool)
    for i, (g, (c, s)) in enumerate(zip(groups, oracle.grouped_gemm(groups))):
        block = got[:g.M, off[i]:off[i] + g.N]
        if g.K == 0:
            assert np.all(block == 0)
        else:
            assert_within_bound(block, c, s, f"kind {kind} group {i} via ldc")
        mask[:g.M, off[i]:off[i] + g.N] = False
    assert np.all(got.view(np.int16)[mask] == CANARY), "a store outside the column blocks"


@pytest.mark.parametrize("mode", ["groups", "n"])
@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("layout", [nv.NVFP4_SF_PREPACKED, nv.NVFP4_SF_ROWMAJOR])
def test_shares_of_one_call_cover_it(mode, world, layout):
    name = "moe_g8_n7168_k2048"
    groups = gen.make_workload(name)
    d = [DeviceGroup(g, layout) for g in groups]
    probs = [x.problem() for x in d]
    for rank in range(world):
        mine = shard.rank_problems(probs, world, rank, mode)
        if mine:
            nv.nvfp4_grouped_gemm(mine)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status()[0] == 0
    for i, (x, (c, s)) in enumerate(zip(d, workload_reference(name))):
        got = x.result()
        assert not np.isnan(got).any(), f"{mode} x{world} group {i}: outputs no share wrote"
        assert_within_bound(got, c, s, f"{mode} x{world} group {i}")
        assert x.guards_intact()
