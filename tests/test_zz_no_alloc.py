"""The no-allocation entry point, nvfp4_grouped_gemm_noalloc, through the C ABI.

It serves callers that must not allocate device memory. Its table lives in a
fixed array inside the library rather than in cached cudaMalloc'd buffers. Its
outputs must match nvfp4_grouped_gemm's on the same inputs, within the
acceptance bound of the other parity tests. That is checked on two calls in a
row with different problem sets, so the second call has to replace the
first call's table in the shared array. This file is named to be collected
last, so a run that stops at the first failure has already run every other
test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
import oracle
from parity import assert_within_bound
import block_scaled_fp4_persistent_gb300 as nv
from gpu_util import DeviceGroup

pytestmark = pytest.mark.gpu


def _noalloc(dgroups):
    probs = (nv.Nvfp4Problem * len(dgroups))(*[d.problem() for d in dgroups])
    stream = torch.cuda.current_stream().cuda_stream
    return nv.lib.nvfp4_grouped_gemm_noalloc(len(dgroups), probs, ctypes.c_void_p(stream))


def test_noalloc_matches_cached_entry_point_on_two_calls_in_a_row():
    nv.lib.nvfp4_grouped_gemm_noalloc.restype = ctypes.c_int
    nv.lib.nvfp4_grouped_gemm_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(nv.Nvfp4Problem), ctypes.c_void_p]
    sets = [gen.make_problem_set(31, [200, 64, 129], [384, 256, 136], [1536, 512, 768]),
            gen.make_problem_set(32, [40, 76, 168, 3], [1024, 512, 264, 8], [2048, 256, 512, 64])]
    # reference outputs from the existing entry point
    ref = []
    for groups in sets:
        d = [DeviceGroup(g) for g in groups]
        nv.nvfp4_grouped_gemm([x.problem() for x in d])
        torch.cuda.synchronize()
        ref.append([x.result().copy() for x in d])
    # two calls in a row of the no-allocation entry point, then one sync
    dev = [[DeviceGroup(g) for g in groups] for groups in sets]
    for d in dev:
        assert _noalloc(d) == nv.NVFP4_OK
    torch.cuda.synchronize()
    for groups, d, r in zip(sets, dev, ref):
        for g, x, c_ref in zip(groups, d, r):
            (_, s), = oracle.grouped_gemm([g])
            got = x.result()
            assert not np.isnan(got).any()
            assert_within_bound(got, c_ref, s, "no-alloc vs cached entry point")
            assert x.guards_intact()


def test_noalloc_rejects_what_it_cannot_hold():
    nv.lib.nvfp4_grouped_gemm_noalloc.restype = ctypes.c_int
    nv.lib.nvfp4_grouped_gemm_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(nv.Nvfp4Problem), ctypes.c_void_p]
    # 16384 x 16384 output tiles' worth of table: far beyond the fixed array; nothing is launched
    big = nv.Nvfp4Problem(1 << 21, 1 << 21, 64, nv.NVFP4_SF_PREPACKED, 256, 256, 256, 256, 256)
    assert nv.lib.nvfp4_grouped_gemm_noalloc(1, (nv.Nvfp4Problem * 1)(big), None) == nv.NVFP4_ERR_TOO_LARGE
    # row-major scales with K % 256 != 0 would need the prepack pass and its workspace
    rowmajor = nv.Nvfp4Problem(128, 128, 320, nv.NVFP4_SF_ROWMAJOR, 256, 256, 256, 256, 256)
    assert nv.lib.nvfp4_grouped_gemm_noalloc(1, (nv.Nvfp4Problem * 1)(rowmajor), None) == nv.NVFP4_ERR_INVALID_ARG


def test_noalloc_reads_row_major_scales_where_k_is_a_multiple_of_256():
    nv.lib.nvfp4_grouped_gemm_noalloc.restype = ctypes.c_int
    nv.lib.nvfp4_grouped_gemm_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(nv.Nvfp4Problem), ctypes.c_void_p]
    groups = gen.make_problem_set(33, [200, 64, 129, 3], [384, 256, 136, 8], [1536, 512, 768, 256])
    # reference: the cached entry point on the same kernel (single CTAs, whole tiles)
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 2)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 0)
    try:
        ref = [DeviceGroup(g) for g in groups]
        nv.nvfp4_grouped_gemm([x.problem() for x in ref])
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 0)
        nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 1)
    d = [DeviceGroup(g, nv.NVFP4_SF_ROWMAJOR) for g in groups]
    assert _noalloc(d) == nv.NVFP4_OK
    torch.cuda.synchronize()
    assert nv.nvfp4_last_launches() == 1
    for g, x, r in zip(groups, d, ref):
        got = x.result()
        assert not np.isnan(got).any() and x.guards_intact()
        # the same scales reach the MMAs by either route: the same bits
        assert np.array_equal(got.view(np.uint16), r.result().view(np.uint16))
