"""M-fusion through the C ABI: groups whose A rows follow one another in memory.

Page 2 of the sources (`_merge_groups`) concatenates the groups' A along M so that
one tensor map serves them all. Here the caller does the concatenating: when
consecutive groups with the same K take their A from consecutive rows of one buffer
(and, for row-major scales read by the kernel, their SFA too), the library encodes
one A map (one SFA map) for the run. The rows of a tile past its group's M then hold
the next group's rows instead of TMA's zero fill. They reach only output rows that
are never stored, so the results must be the same bits as with separate buffers.
M-fusion applies to the CTA-pair kernel, which serves the many-group sets; the
single-CTA kernel keeps one map per group and must give the same bits from the
concatenated buffers too. Checked for both kernel kinds and both scale layouts,
with ragged M, against the same data in separate buffers with fusion off, and
against the oracle's bound.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity import assert_within_bound
import block_scaled_fp4_persistent_gb300 as nv
from gpu_util import DeviceGroup, run, workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for opt, val in [(nv.NVFP4_OPT_CTA_PAIR, 0), (nv.NVFP4_OPT_M_FUSION, 1), (nv.NVFP4_OPT_SPLIT_TAIL, 1)]:
        nv.nvfp4_set_option(opt, val)


class FusedView:
    """The groups of `dgroups` with A (and row-major SFA) moved into one buffer per
    run: run r holds the groups of runs[r] back to back. B, SFB and a fresh C stay
    per group. Groups in no run keep their own buffers."""

    def __init__(self, dgroups, runs):
        self.d = dgroups
        self.a_ptr = {i: d.A.data_ptr() for i, d in enumerate(dgroups)}
        self.sfa_ptr = {i: d.SFA.data_ptr() for i, d in enumerate(dgroups)}
        self.keep = []
        for run_ in runs:
            a_cat = torch.cat([dgroups[i].A.reshape(-1) for i in run_])
            self.keep.append(a_cat)
            off = 0
            for i in run_:
                self.a_ptr[i] = a_cat.data_ptr() + off
                off += dgroups[i].A.numel()
            if dgroups[run_[0]].sf_layout == nv.NVFP4_SF_ROWMAJOR:
                s_cat = torch.cat([dgroups[i].SFA.reshape(-1) for i in run_])
                self.keep.append(s_cat)
                off = 0
                for i in run_:
                    self.sfa_ptr[i] = s_cat.data_ptr() + off
                    off += dgroups[i].SFA.numel()
        self.C = [torch.full((d.M, d.N), float("nan"), dtype=torch.float16, device="cuda") for d in dgroups]

    def problems(self):
        return [nv.Nvfp4Problem(d.M, d.N, d.K, d.sf_layout, self.a_ptr[i], d.B.data_ptr(), self.sfa_ptr[i],
                                d.SFB.data_ptr(), self.C[i].data_ptr()) for i, d in enumerate(self.d)]

    def results(self):
        return [c.cpu().numpy() for c in self.C]


def _reference(dgroups):
    nv.nvfp4_set_option(nv.NVFP4_OPT_M_FUSION, 0)
    run(dgroups)
    assert nv.nvfp4_last_a_maps() == len(dgroups)
    nv.nvfp4_set_option(nv.NVFP4_OPT_M_FUSION, 1)
    return [d.result().copy() for d in dgroups]


def _fused(view, a_maps):
    nv.nvfp4_grouped_gemm(view.problems())
    torch.cuda.synchronize()
    status, detail = nv.nvfp4_device_status(None)
    assert status == 0, f"device status {status}: {detail}"
    assert nv.nvfp4_last_a_maps() == a_maps
    return view.results()


@pytest.mark.parametrize("split", [1, 2], ids=["split-single", "split-all"])
@pytest.mark.parametrize("pair", [1, 2], ids=["pairs", "single"])
@pytest.mark.parametrize("layout", [nv.NVFP4_SF_PREPACKED, nv.NVFP4_SF_ROWMAJOR], ids=["prepacked", "rowmajor"])
def test_concatenated_a_is_one_map_and_the_same_bits(pair, layout, split):
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, split)  # 2: split tails on pairs too, items cut along K
    # one K (1536: whole 256-wide stages, so row-major scales are read directly), ragged M, mixed N
    groups = gen.make_problem_set(41, [200, 64, 129, 3, 256, 77], [384, 256, 136, 8, 512, 264], [1536] * 6)
    dgroups = [DeviceGroup(g, layout) for g in groups]
    ref = _reference(dgroups)
    # M-fusion is for the pair kernel; single CTAs keep one map per group
    got = _fused(FusedView(dgroups, [list(range(len(groups)))]), 1 if pair == 1 else len(groups))
    oref = oracle.grouped_gemm(groups)
    for i, (g, r, c, (c_ref, s_ref)) in enumerate(zip(groups, ref, got, oref)):
        assert not np.isnan(c).any(), f"group {i}: unwritten outputs"
        assert np.array_equal(c.view(np.uint16), r.view(np.uint16)), f"group {i}: fused A changed the bits"
        assert_within_bound(c, c_ref, s_ref, f"fused group {i}")


def test_runs_break_where_rows_or_k_do_not_follow():
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 1)
    # K changes between groups 2 and 3; group 2's A lives in a buffer of its own
    groups = gen.make_problem_set(42, [130, 96, 40, 200, 17], [256, 128, 264, 136, 512], [1024, 1024, 1024, 512, 512])
    dgroups = [DeviceGroup(g) for g in groups]
    ref = _reference(dgroups)
    # runs {0, 1}, {2}, {3, 4}: three A maps
    got = _fused(FusedView(dgroups, [[0, 1], [3, 4]]), 3)
    for i, (r, c) in enumerate(zip(ref, got)):
        assert np.array_equal(c.view(np.uint16), r.view(np.uint16)), f"group {i}"
    # the same buffers with fusion off: one map per group, the same bits
    nv.nvfp4_set_option(nv.NVFP4_OPT_M_FUSION, 0)
    view = FusedView(dgroups, [[0, 1], [3, 4]])
    got = _fused(view, len(groups))
    for i, (r, c) in enumerate(zip(ref, got)):
        assert np.array_equal(c.view(np.uint16), r.view(np.uint16)), f"group {i}, fusion off"
    # one run across a change of K is not fused: {0, 1, 2} and {3, 4} stay apart
    nv.nvfp4_set_option(nv.NVFP4_OPT_M_FUSION, 1)
    got = _fused(FusedView(dgroups, [[0, 1, 2, 3, 4]]), 2)
    for i, (r, c) in enumerate(zip(ref, got)):
        assert np.array_equal(c.view(np.uint16), r.view(np.uint16)), f"group {i}, across K"


@pytest.mark.parametrize("layout", [nv.NVFP4_SF_PREPACKED, nv.NVFP4_SF_ROWMAJOR], ids=["prepacked", "rowmajor"])
@pytest.mark.parametrize("name", ["moe_g8_n7168_k2048", "moe_g8_n4096_k7168"])
def test_full_size_moe_with_concatenated_a(name, layout):
    # the MoE layout: every expert's tokens are consecutive rows of one activation tensor
    groups = gen.make_workload(name)
    dgroups = [DeviceGroup(g, layout) for g in groups]
    ref = _reference(dgroups)  # separate buffers, one map per group, automatic kernel choice (pairs)
    got = _fused(FusedView(dgroups, [list(range(len(groups)))]), 1)
    for i, (g, r, c, (c_ref, s_ref)) in enumerate(zip(groups, ref, got, workload_reference(name))):
        assert np.array_equal(c.view(np.uint16), r.view(np.uint16)), f"{name} group {i}"
        assert_within_bound(c, c_ref, s_ref, f"{name} group {i}, fused")
