"""Randomised parity through the C ABI: many small problem sets, every output against the oracle.

Each case draws (from a fixed seed) a problem set of 1-5 groups with ragged M, N a multiple of 8
and K a multiple of 64, a scale layout (prepacked; row-major, read in the kernel where K % 256 = 0
and through the prepack launch otherwise), a kernel kind (automatic, CTA pairs, single CTAs), a
split-tail mode, and whether the groups' A rows sit back to back in one buffer (M-fusion on pairs).
Every output must lie within the acceptance bound, every output must be written, and the guard
bands around C must be intact.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity import assert_within_bound
import block_scaled_fp4_persistent_gb300 as nv
from gpu_util import DeviceGroup

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for opt, val in [(nv.NVFP4_OPT_CTA_PAIR, 0), (nv.NVFP4_OPT_SPLIT_TAIL, 1), (nv.NVFP4_OPT_M_FUSION, 1)]:
        nv.nvfp4_set_option(opt, val)


def _draw(rng):
    g = int(rng.integers(1, 6))
    K = int(rng.integers(1, 25)) * 64
    Ms = [int(rng.integers(1, 257)) for _ in range(g)]
    Ns = [int(rng.integers(1, 65)) * 8 for _ in range(g)]
    # mixed K across groups now and then (no fusion across a change of K)
    Ks = [K if rng.random() < 0.8 else int(rng.integers(1, 25)) * 64 for _ in range(g)]
    return Ms, Ns, Ks


@pytest.mark.parametrize("case", range(CASES))
def test_random_problem_sets_match_oracle(case):
    rng = np.random.default_rng(1000 + case)
    Ms, Ns, Ks = _draw(rng)
    layout = nv.NVFP4_SF_ROWMAJOR if rng.random() < 0.5 else nv.NVFP4_SF_PREPACKED
    pair = int(rng.integers(0, 3))
    split = int(rng.integers(0, 3))
    concat = rng.random() < 0.5
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, split)
    groups = gen.make_problem_set(5000 + case, Ms, Ns, Ks)
    d = [DeviceGroup(g, layout) for g in groups]
    a_ptr = [x.A.data_ptr() for x in d]
    sfa_ptr = [x.SFA.data_ptr() for x in d]
    keep = []
    if concat:
        # A (and row-major SFA) of all groups back to back in one buffer
        a_cat = torch.cat([x.A.reshape(-1) for x in d])
        keep.append(a_cat)
        off = 0
        for i, x in enumerate(d):
            a_ptr[i] = a_cat.data_ptr() + off
            off += x.A.numel()
        if layout == nv.NVFP4_SF_ROWMAJOR:
            # back to back where the sizes keep the 16-byte alignment the ABI asks of
            # every pointer, else padded to it (which ends a run: those rows do not follow)
            offs, off = [], 0
            for x in d:
                offs.append(off)
                off = (off + x.SFA.numel() + 15) // 16 * 16
            s_cat = torch.zeros(off, dtype=torch.uint8, device="cuda")
            keep.append(s_cat)
            for i, x in enumerate(d):
                s_cat[offs[i]:offs[i] + x.SFA.numel()].copy_(x.SFA.reshape(-1))
                sfa_ptr[i] = s_cat.data_ptr() + offs[i]
    probs = [nv.Nvfp4Problem(x.M, x.N, x.K, x.sf_layout, a_ptr[i], x.B.data_ptr(), sfa_ptr[i], x.SFB.data_ptr(),
                             x.C.data_ptr()) for i, x in enumerate(d)]
    nv.nvfp4_grouped_gemm(probs)
    torch.cuda.synchronize()
    status, detail = nv.nvfp4_device_status(None)
    what = f"case {case}: M={Ms} N={Ns} K={Ks} layout={layout} pair={pair} split={split} concat={concat}"
    assert status == 0, f"{what}: device status {status} {detail}"
    for i, ((c_ref, s_ref), x) in enumerate(zip(oracle.grouped_gemm(groups), d)):
        got = x.result()
        assert not np.isnan(got).any(), f"{what} group {i}: unwritten outputs"
        assert x.guards_intact(), f"{what} group {i}: guard band"
        assert_within_bound(got, c_ref, s_ref, f"{what} group {i}")
