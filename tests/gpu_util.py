"""Helpers for the GPU tests: upload generated groups, call the library through the
C ABI, and check canary guard bands around every output buffer."""
import functools

import numpy as np
import torch

import gen
import oracle

import block_scaled_fp4_persistent_gb300 as nv

GUARD = 2048          # fp16 elements of guard band before and after each C (4 KB)
CANARY = 0x7E5A       # a NaN pattern that no kernel store produces
FILL = 0x7E00         # the NaN that fills C before a call, to catch unwritten outputs


class DeviceGroup:
    def __init__(self, g, sf_layout=nv.NVFP4_SF_PREPACKED, device="cuda"):
        self.g = g
        self.M, self.N, self.K = g.M, g.N, g.K
        self.A = torch.from_numpy(np.ascontiguousarray(g.A)).to(device)
        self.B = torch.from_numpy(np.ascontiguousarray(g.B)).to(device)
        sfa = torch.from_numpy(np.ascontiguousarray(g.SFA)).to(device)
        sfb = torch.from_numpy(np.ascontiguousarray(g.SFB)).to(device)
        if sf_layout == nv.NVFP4_SF_PREPACKED and g.K > 0 and g.M > 0 and g.N > 0:
            self.SFA = nv.prepack_scales(sfa, g.K)
            self.SFB = nv.prepack_scales(sfb, g.K)
        else:
            self.SFA, self.SFB = sfa, sfb
        self.sf_layout = sf_layout
        n = g.M * g.N
        self.buf = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.int16, device=device).view(torch.float16)
        self.C = self.buf[GUARD:GUARD + n].view(g.M, g.N)
        self.reset()

    def reset(self):
        self.C.view(torch.int16).fill_(FILL)

    def problem(self):
        M, N, K = self.M, self.N, self.K
        ptr = lambda t: t.data_ptr() if t.numel() else 0
        return nv.Nvfp4Problem(M, N, K, self.sf_layout, ptr(self.A), ptr(self.B), ptr(self.SFA), ptr(self.SFB),
                               ptr(self.C) if M * N else 0)

    def result(self) -> np.ndarray:
        return self.C.cpu().numpy()

    def guards_intact(self) -> bool:
        b = self.buf.view(torch.int16)
        n = self.M * self.N
        return bool((b[:GUARD] == CANARY).all()) and bool((b[GUARD + n:] == CANARY).all())


def run(dgroups, stream=None):
    nv.nvfp4_grouped_gemm([d.problem() for d in dgroups], stream)
    torch.cuda.synchronize()
    status, detail = nv.nvfp4_device_status(stream)
    assert status == 0, f"device status {status}: {detail}"


@functools.lru_cache(maxsize=None)
def workload_reference(name):
    """The oracle's (C, S) for every output of a named workload, computed once per test
    session (the full-size sets take the oracle about a second or two on the host's cores)."""
    return oracle.grouped_gemm(gen.make_workload(name))
