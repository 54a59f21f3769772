"""The kernel's bounded waits: a wait that can never complete ends with an error
status and the GPU stays usable.

The failure is made on the host. NVFP4_OPT_FAULT_SKIP_LOAD tells the producer of
CTA 0 to arm one k-stage's barrier without issuing its copies, so the MMA
warp's wait on that stage never completes. With a 20 ms bound, the kernel must
record NVFP4_ERR_TIMEOUT, wait for its own copies in flight, free its TMEM and
return. There is no trap and no fault.
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


# Which waiting role reports first is not fixed: the MMA issuer waits on the starved slot, the
# producer waits for that slot to be freed (long K) or for its own copies before exit (short K),
# and try_wait suspends for hardware-chosen intervals between the checks of the bound.
# The status and the recovery are what the test pins.
CASES = [([128], [128], [4096]), ([64, 128], [512, 512], [512, 512])]


@pytest.mark.parametrize("pair", [1, 2, 3, 4])
@pytest.mark.parametrize("Ms,Ns,Ks", CASES)
def test_wait_timeout_reports_and_recovers(Ms, Ns, Ks, pair):
    groups = gen.make_problem_set(1, Ms, Ns, Ks)
    d = [DeviceGroup(g) for g in groups]
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    try:
        nv.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 20000)
        nv.nvfp4_set_option(nv.NVFP4_OPT_FAULT_SKIP_LOAD, 0)
        nv.nvfp4_grouped_gemm([x.problem() for x in d])
        status, detail = nv.nvfp4_device_status()
        assert status == nv.NVFP4_ERR_TIMEOUT, (status, detail)
        assert detail[0] == nv.NVFP4_ERR_TIMEOUT and detail[1] in (0, 1, 2, 3, 4), detail
        assert nv.nvfp4_device_status()[0] == 0  # reading cleared it
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_FAULT_SKIP_LOAD, -1)
        nv.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 2000000)
    try:
        for x in d:
            x.reset()
        nv.nvfp4_grouped_gemm([x.problem() for x in d])
        torch.cuda.synchronize()
        assert nv.nvfp4_device_status()[0] == 0
        for g, x, (c, s) in zip(groups, d, oracle.grouped_gemm(groups)):
            assert_within_bound(x.result(), c, s, "after recovery")
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 0)
