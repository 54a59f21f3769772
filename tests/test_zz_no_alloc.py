"""The no-allocation entry point, nvfp4_grouped_gemm_noalloc, through the C ABI.

It serves callers that must not allocate device memory (code inside a custom
allocator or an out-of-memory handler, or a runtime that owns every byte of
device memory). Its table lives in a fixed array inside the library rather than
in cached cudaMalloc'd buffers. Its outputs are checked against the oracle,
output by output within the acceptance bound of every other parity test, on two
calls in a row with different problem sets: the second call has to replace the
first call's table in the shared array. Where the cached entry point runs the
same kernel on the same schedule, the two must also agree bit for bit.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
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


def _noalloc(dgroups, stream=None):
    return nv.nvfp4_grouped_gemm_noalloc([d.problem() for d in dgroups], stream, check=False)


def _check_oracle(groups, dgroups, what):
    for i, (g, x, (c, s)) in enumerate(zip(groups, dgroups, oracle.grouped_gemm(groups))):
        got = x.result()
        assert not np.isnan(got).any(), f"{what} group {i}: unwritten outputs"
        assert_within_bound(got, c, s, f"{what} group {i}")
        assert x.guards_intact(), f"{what} group {i}: store outside C"


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    sets = [gen.make_problem_set(31, [200, 64, 129], [384, 256, 136], [1536, 512, 768]),
            gen.make_problem_set(32, [40, 76, 168, 3], [1024, 512, 264, 8], [2048, 256, 512, 64])]
    # two calls in a row of the no-allocation entry point, then one sync
    dev = [[DeviceGroup(g) for g in groups] for groups in sets]
    for d in dev:
        assert _noalloc(d) == nv.NVFP4_OK
    torch.cuda.synchronize()
    assert nv.nvfp4_noalloc_status()[0] == nv.NVFP4_OK
    for k, (groups, d) in enumerate(zip(sets, dev)):
        _check_oracle(groups, d, f"no-alloc call {k}")


def test_noalloc_same_bits_as_the_cached_entry_point_on_the_same_kernel():
    groups = gen.make_problem_set(34, [200, 64, 129, 3], [384, 256, 136, 8], [1536, 512, 768, 256])
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 2)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 0)
    try:
        ref = [DeviceGroup(g) for g in groups]
        nv.nvfp4_grouped_gemm([x.problem() for x in ref])
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 0)
        nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 1)
    d = [DeviceGroup(g) for g in groups]
    assert _noalloc(d) == nv.NVFP4_OK
    torch.cuda.synchronize()
    _check_oracle(groups, d, "no-alloc")
    for x, r in zip(d, ref):
        assert np.array_equal(x.result().view(np.uint16), r.result().view(np.uint16))


def test_noalloc_rejects_what_it_cannot_hold():
    # 16384 x 16384 output tiles' worth of table: far beyond the fixed array; nothing is launched
    big = nv.Nvfp4Problem(1 << 21, 1 << 21, 64, nv.NVFP4_SF_PREPACKED, 256, 256, 256, 256, 256)
    assert nv.nvfp4_grouped_gemm_noalloc([big], None, check=False) == nv.NVFP4_ERR_TOO_LARGE
    # row-major scales with K % 256 != 0 would need the prepack pass and its workspace
    rowmajor = nv.Nvfp4Problem(128, 128, 320, nv.NVFP4_SF_ROWMAJOR, 256, 256, 256, 256, 256)
    assert nv.nvfp4_grouped_gemm_noalloc([rowmajor], None, check=False) == nv.NVFP4_ERR_INVALID_ARG


def test_noalloc_reads_row_major_scales_where_k_is_a_multiple_of_256():
    groups = gen.make_problem_set(33, [200, 64, 129, 3], [384, 256, 136, 8], [1536, 512, 768, 256])
    d = [DeviceGroup(g, nv.NVFP4_SF_ROWMAJOR) for g in groups]
    assert _noalloc(d) == nv.NVFP4_OK
    torch.cuda.synchronize()
    assert nv.nvfp4_last_launches() == 1
    _check_oracle(groups, d, "no-alloc, row-major scales")


def test_noalloc_refuses_a_capturing_stream():
    groups = gen.make_problem_set(35, [64], [128], [256])
    d = [DeviceGroup(g) for g in groups]
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    rc = None
    with torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        rc = _noalloc(d, s)
    assert rc == nv.NVFP4_ERR_CAPTURE
    torch.cuda.synchronize()
    # outside a capture the same call runs
    assert _noalloc(d) == nv.NVFP4_OK
    torch.cuda.synchronize()
    _check_oracle(groups, d, "no-alloc after a refused capture")


def test_noalloc_reports_a_timeout_and_recovers():
    # The producer of CTA 0 skips one stage's copies, so a bounded wait runs out; the
    # status must come back through nvfp4_noalloc_status, without any allocation.
    groups = gen.make_problem_set(36, [64, 128], [512, 512], [512, 512])
    d = [DeviceGroup(g) for g in groups]
    nv.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 20000)
    nv.nvfp4_set_option(nv.NVFP4_OPT_FAULT_SKIP_LOAD, 0)
    try:
        assert _noalloc(d) == nv.NVFP4_OK
        status, detail = nv.nvfp4_noalloc_status()
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_FAULT_SKIP_LOAD, -1)
        nv.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 2000000)
    assert status == nv.NVFP4_ERR_TIMEOUT, (status, detail)
    assert detail[0] == nv.NVFP4_ERR_TIMEOUT and detail[1] in (0, 1, 2, 3, 4), detail
    assert nv.nvfp4_noalloc_status()[0] == nv.NVFP4_OK  # reading cleared it
    for x in d:
        x.reset()
    assert _noalloc(d) == nv.NVFP4_OK
    assert nv.nvfp4_noalloc_status()[0] == nv.NVFP4_OK
    _check_oracle(groups, d, "no-alloc after a timeout")
