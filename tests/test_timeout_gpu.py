"""The kernel's bounded waits: a wait that can never complete ends with an error
status and the GPU stays usable.

The failure is made on the host. NVFP4_OPT_FAULT_SKIP_LOAD tells the producer of
CTA 0 to arm one k-stage's barrier without issuing its copies, so the MMA
warp's wait on that stage never completes. With a 20 ms bound, the kernel must
record NVFP4_ERR_TIMEOUT (role 1 = MMA issuer, k-stage 0), wait for its own
copies in flight, free its TMEM and return. There is no trap and no fault.
The next normal launch must then give correct results.
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


# (Ms, Ns, Ks, roles): with one long-K tile (16 k-stages), the MMA issuer's wait on k-stage 0 runs
# out first (role 1). With two k-stages per tile the producer has already reached its final wait
# for its own copies, so either that wait (role 3) or the MMA issuer's reports first.
CASES = [([128], [128], [4096], {1}), ([64, 128], [512, 512], [512, 512], {1, 3})]


@pytest.mark.parametrize("Ms,Ns,Ks,roles", CASES)
def test_wait_timeout_reports_and_recovers(Ms, Ns, Ks, roles):
    groups = gen.make_problem_set(1, Ms, Ns, Ks)
    d = [DeviceGroup(g) for g in groups]
    try:
        nv.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 20000)
        nv.nvfp4_set_option(nv.NVFP4_OPT_FAULT_SKIP_LOAD, 0)
        nv.nvfp4_grouped_gemm([x.problem() for x in d])
        status, detail = nv.nvfp4_device_status()
        assert status == nv.NVFP4_ERR_TIMEOUT, (status, detail)
        assert detail[1] in roles and detail[3] == 0, detail  # k-stage / ring slot 0
        assert nv.nvfp4_device_status()[0] == 0  # reading cleared it
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_FAULT_SKIP_LOAD, -1)
        nv.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 2000000)
    for x in d:
        x.reset()
    nv.nvfp4_grouped_gemm([x.problem() for x in d])
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status()[0] == 0
    for g, x, (c, s) in zip(groups, d, oracle.grouped_gemm(groups)):
        assert_within_bound(x.result(), c, s, "after recovery")
