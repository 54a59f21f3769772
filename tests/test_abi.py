"""The C ABI without a GPU: the library loads, exports every declared symbol, and
rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def nv():
    from block_scaled_fp4_persistent_gb300 import _build
    _build.build()
    import block_scaled_fp4_persistent_gb300 as nv
    return nv


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(nvfp4_\w+)\s*\(", text, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(nv):
    names = declared_functions()
    assert {"nvfp4_grouped_gemm", "nvfp4_prepack_scales", "nvfp4_prepacked_scale_bytes",
            "nvfp4_device_status", "nvfp4_status_string", "nvfp4_release"} <= set(names)
    lib = ctypes.CDLL(nv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_no_driver_or_runtime_link(nv):
    # cudart is linked statically and the driver is reached through the runtime,
    # so the library loads (as here) on a machine without a GPU driver
    import shutil
    import subprocess
    if not shutil.which("ldd"):
        pytest.skip("no ldd")
    out = subprocess.run(["ldd", nv.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcudart" not in out and "libcuda.so" not in out


def test_prepacked_scale_bytes(nv):
    assert nv.nvfp4_prepacked_scale_bytes(0, 64) == 0
    assert nv.nvfp4_prepacked_scale_bytes(1, 64) == 128 * 4
    assert nv.nvfp4_prepacked_scale_bytes(128, 256) == 128 * 16
    assert nv.nvfp4_prepacked_scale_bytes(129, 7168) == 256 * 448
    assert nv.nvfp4_prepacked_scale_bytes(40, 2048) == 128 * 128


def test_status_strings(nv):
    for code in [0, -1, -2, -3, -4, -5, -6, -7]:
        s = nv.nvfp4_status_string(code)
        assert s and s != "unknown status"
    assert nv.nvfp4_status_string(-99) == "unknown status"


def _p(nv, M=128, N=128, K=256, A=256, B=256, SFA=256, SFB=256, C=256, layout=0):
    return nv.Nvfp4Problem(M, N, K, layout, A, B, SFA, SFB, C)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), -1), (dict(N=-1), -1), (dict(K=-64), -1), (dict(layout=7), -1),
    (dict(C=0), -1), (dict(A=0), -1), (dict(SFB=0), -1),
    (dict(K=96), -2), (dict(N=100), -2), (dict(A=264), -2), (dict(C=2), -2), (dict(SFA=8), -2),
    (dict(M=1 << 24), -6), (dict(K=1 << 24), -6),
])
def test_host_argument_checks(nv, kw, code):
    rc = nv.lib.nvfp4_grouped_gemm(1, (nv.Nvfp4Problem * 1)(_p(nv, **kw)), None)
    assert rc == code


def test_trivial_calls_do_not_touch_cuda(nv):
    assert nv.lib.nvfp4_grouped_gemm(0, None, None) == 0
    assert nv.lib.nvfp4_grouped_gemm(-1, None, None) == -1
    assert nv.lib.nvfp4_grouped_gemm(1, None, None) == -1
    assert nv.lib.nvfp4_prepack_scales(None, 0, 64, None, None) == 0
    assert nv.lib.nvfp4_prepack_scales(None, 4, 40, None, None) == -1  # K % 16
    assert nv.lib.nvfp4_prepack_scales(None, 4, 64, None, None) == -1  # null pointers
    assert nv.lib.nvfp4_prepack_scales(8, 4, 64, 256, None) == -2
    assert nv.nvfp4_last_kernel() == "none"  # nothing launched in a process without a GPU
    assert nv.nvfp4_last_launches() == 0
    assert nv.nvfp4_last_a_maps() == 0


def test_options(nv):
    lib = nv.lib
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_STAGES, 5) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_STAGES, 4) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_STAGES, 3) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_BLOCK_N, 64) == -1
    assert lib.nvfp4_set_option(99, 1) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 5) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 4) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, -1) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_WAIT_TIMEOUT_US, 0) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_SF_DIRECT, 2) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_SF_DIRECT, -1) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_PDL, 2) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_M_FUSION, 2) == -1
    assert lib.nvfp4_set_option(nv.NVFP4_OPT_M_FUSION, -1) == -1
    for opt, val in [(nv.NVFP4_OPT_STAGES, 2), (nv.NVFP4_OPT_STAGES, 0), (nv.NVFP4_OPT_BLOCK_N, 256),
                     (nv.NVFP4_OPT_BLOCK_N, 128), (nv.NVFP4_OPT_MAX_CTAS, 3),
                     (nv.NVFP4_OPT_MAX_CTAS, 0), (nv.NVFP4_OPT_WAIT_TIMEOUT_US, 2000000),
                     (nv.NVFP4_OPT_FAULT_SKIP_LOAD, -1), (nv.NVFP4_OPT_BLOCK_N, 0),
                     (nv.NVFP4_OPT_CTA_PAIR, 1), (nv.NVFP4_OPT_CTA_PAIR, 2), (nv.NVFP4_OPT_CTA_PAIR, 3),
                     (nv.NVFP4_OPT_CTA_PAIR, 4), (nv.NVFP4_OPT_CTA_PAIR, 0),
                     (nv.NVFP4_OPT_SPLIT_TAIL, 2), (nv.NVFP4_OPT_SPLIT_TAIL, 3), (nv.NVFP4_OPT_SPLIT_TAIL, 0),
                     (nv.NVFP4_OPT_SPLIT_TAIL, 1),
                     (nv.NVFP4_OPT_SF_DIRECT, 0), (nv.NVFP4_OPT_SF_DIRECT, 1), (nv.NVFP4_OPT_PDL, 1),
                     (nv.NVFP4_OPT_PDL, 0), (nv.NVFP4_OPT_M_FUSION, 0), (nv.NVFP4_OPT_M_FUSION, 1)]:
        assert lib.nvfp4_set_option(opt, val) == 0
