"""Python binding of libnvfp4gg.so, the grouped NVFP4 block-scaled GEMM for GB300 (sm_103a).

This module only marshals arguments. It converts them to the C ABI declared in
``include/nvfp4_grouped_gemm.h`` and calls the library; every step of the
computation runs in the library's CUDA kernels. PyTorch supplies device memory
and streams. The library has no fallback path: if ``libnvfp4gg.so`` has not
been built, the first call raises ImportError. Build it with
``block_scaled_fp4_persistent_gb300._build.build()`` or
``__graft_entry__.build()``.

Names match the C ABI: ``nvfp4_grouped_gemm``, ``nvfp4_prepack_scales``, ``nvfp4_prepack_scales_batch``,
``nvfp4_prepacked_scale_bytes``, ``nvfp4_device_status``,
``nvfp4_status_string``, ``nvfp4_last_cuda_error``, ``nvfp4_last_kernel``, ``nvfp4_last_launches``,
``nvfp4_last_a_maps``, ``nvfp4_set_option``, ``nvfp4_release``,
``nvfp4_grouped_gemm_noalloc`` and ``nvfp4_noalloc_status``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, List, Optional, Sequence, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4gg.so")

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = -1
NVFP4_ERR_ALIGNMENT = -2
NVFP4_ERR_UNSUPPORTED_DEVICE = -3
NVFP4_ERR_CUDA = -4
NVFP4_ERR_TIMEOUT = -5
NVFP4_ERR_TOO_LARGE = -6
NVFP4_ERR_CAPTURE = -7

NVFP4_SF_PREPACKED = 0
NVFP4_SF_ROWMAJOR = 1

NVFP4_OPT_BLOCK_N = 1
NVFP4_OPT_STAGES = 2
NVFP4_OPT_MAX_CTAS = 3
NVFP4_OPT_WAIT_TIMEOUT_US = 4
NVFP4_OPT_FAULT_SKIP_LOAD = 5
NVFP4_OPT_PREFETCH_STAGES = 6
NVFP4_OPT_SPLIT_TAIL = 7
NVFP4_OPT_CTA_PAIR = 8
NVFP4_OPT_SF_DIRECT = 9
NVFP4_OPT_PDL = 10
NVFP4_OPT_M_FUSION = 11


class Nvfp4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {nvfp4_status_string(code)} ({code})"
                         + (f", cudaError {nvfp4_last_cuda_error()}" if code == NVFP4_ERR_CUDA else ""))


class Nvfp4Problem(ctypes.Structure):
    """One group: sizes, layout of the scales, and device pointers (see the C header)."""

    _fields_ = [
        ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("sf_layout", ctypes.c_int32),
        ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("SFA", ctypes.c_void_p), ("SFB", ctypes.c_void_p),
        ("C", ctypes.c_void_p),
        ("ldc", ctypes.c_int32),       # elements between rows of C; 0 means N
        ("reserved", ctypes.c_int32),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: the CUDA library has not been built. "
            "Run block_scaled_fp4_persistent_gb300._build.build() (needs nvcc).")
    lib = ctypes.CDLL(LIB_PATH)
    lib.nvfp4_grouped_gemm.restype = ctypes.c_int
    lib.nvfp4_grouped_gemm.argtypes = [ctypes.c_int, ctypes.POINTER(Nvfp4Problem), ctypes.c_void_p]
    lib.nvfp4_prepacked_scale_bytes.restype = ctypes.c_size_t
    lib.nvfp4_prepacked_scale_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.nvfp4_prepack_scales.restype = ctypes.c_int
    lib.nvfp4_prepack_scales.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.nvfp4_prepack_scales_batch.restype = ctypes.c_int
    lib.nvfp4_prepack_scales_batch.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
                                               ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                               ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
    lib.nvfp4_device_status.restype = ctypes.c_int
    lib.nvfp4_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int32)]
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_status_string.argtypes = [ctypes.c_int]
    lib.nvfp4_last_cuda_error.restype = ctypes.c_int
    lib.nvfp4_last_cuda_error.argtypes = []
    lib.nvfp4_last_kernel.restype = ctypes.c_char_p
    lib.nvfp4_last_kernel.argtypes = []
    lib.nvfp4_last_launches.restype = ctypes.c_int
    lib.nvfp4_last_launches.argtypes = []
    lib.nvfp4_last_a_maps.restype = ctypes.c_int
    lib.nvfp4_last_a_maps.argtypes = []
    lib.nvfp4_set_option.restype = ctypes.c_int
    lib.nvfp4_set_option.argtypes = [ctypes.c_int, ctypes.c_int64]
    lib.nvfp4_release.restype = None
    lib.nvfp4_release.argtypes = []
    lib.nvfp4_grouped_gemm_noalloc.restype = ctypes.c_int
    lib.nvfp4_grouped_gemm_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(Nvfp4Problem), ctypes.c_void_p]
    lib.nvfp4_noalloc_status.restype = ctypes.c_int
    lib.nvfp4_noalloc_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int32)]
    return lib


_lib = None


def _get() -> ctypes.CDLL:
    """The loaded library. The first call loads it, and raises ImportError if it was never built."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def __getattr__(name):
    if name == "lib":
        return _get()
    raise AttributeError(name)


def _stream_handle(stream) -> Optional[int]:
    """A raw cudaStream_t from an int, a torch.cuda.Stream or None (torch's current stream)."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, what: str) -> int:
    if code != NVFP4_OK:
        raise Nvfp4Error(code, what)
    return code


# ---------------------------------------------------------------- C ABI names --

def nvfp4_grouped_gemm(probs: Sequence[Nvfp4Problem], stream=None, check: bool = True) -> int:
    """One grouped GEMM launch over ``probs``. Raises Nvfp4Error unless check is False."""
    arr = (Nvfp4Problem * max(1, len(probs)))(*probs)
    rc = _get().nvfp4_grouped_gemm(len(probs), arr, _stream_handle(stream))
    return _check(rc, "nvfp4_grouped_gemm") if check else rc


def nvfp4_prepacked_scale_bytes(rows: int, K: int) -> int:
    return int(_get().nvfp4_prepacked_scale_bytes(rows, K))


def nvfp4_prepack_scales(sf_rowmajor_ptr: int, rows: int, K: int, sf_blocked_ptr: int, stream=None,
                         check: bool = True) -> int:
    rc = _get().nvfp4_prepack_scales(sf_rowmajor_ptr, rows, K, sf_blocked_ptr, _stream_handle(stream))
    return _check(rc, "nvfp4_prepack_scales") if check else rc


def nvfp4_prepack_scales_batch(src_ptrs: Sequence[int], rows: Sequence[int], Ks: Sequence[int],
                               dst_ptrs: Sequence[int], stream=None, check: bool = True) -> int:
    """Prepack of several operands in one launch (see the C header)."""
    n = len(src_ptrs)
    if not (len(rows) == len(Ks) == len(dst_ptrs) == n):
        raise ValueError("nvfp4_prepack_scales_batch: the four lists must have the same length")
    m = max(1, n)
    src = (ctypes.c_void_p * m)(*src_ptrs)
    dst = (ctypes.c_void_p * m)(*dst_ptrs)
    r = (ctypes.c_int * m)(*rows)
    k = (ctypes.c_int * m)(*Ks)
    rc = _get().nvfp4_prepack_scales_batch(n, src, r, k, dst, _stream_handle(stream))
    return _check(rc, "nvfp4_prepack_scales_batch") if check else rc


def nvfp4_device_status(stream=None) -> Tuple[int, List[int]]:
    """(status, [code, role, item, stage]) of the device error word; reading clears it."""
    st = ctypes.c_int(0)
    detail = (ctypes.c_int32 * 4)()
    _check(_get().nvfp4_device_status(_stream_handle(stream), ctypes.byref(st), detail), "nvfp4_device_status")
    return st.value, list(detail)


def nvfp4_status_string(code: int) -> str:
    return _get().nvfp4_status_string(code).decode()


def nvfp4_last_cuda_error() -> int:
    return int(_get().nvfp4_last_cuda_error())


def nvfp4_last_kernel() -> str:
    return _get().nvfp4_last_kernel().decode()


def nvfp4_last_launches() -> int:
    return _get().nvfp4_last_launches()


def nvfp4_last_a_maps() -> int:
    return _get().nvfp4_last_a_maps()


def nvfp4_set_option(option: int, value: int) -> None:
    _check(_get().nvfp4_set_option(option, int(value)), "nvfp4_set_option")


def nvfp4_release() -> None:
    _get().nvfp4_release()


# ------------------------------------------------------- torch tensor helpers --

def problem(A, B, SFA, SFB, C, sf_layout: int = NVFP4_SF_PREPACKED) -> Nvfp4Problem:
    """An Nvfp4Problem from CUDA tensors. A: uint8 [M, K/2]; B: uint8 [N, K/2];
    SFA/SFB: uint8 scale bytes in `sf_layout`; C: fp16 [M, N], dense, or a column
    block of a wider row-major matrix (its row stride becomes ldc). The caller keeps
    the tensors alive until the launch has run."""
    M, N = C.shape
    K = A.shape[1] * 2 if A.dim() == 2 else 0
    ldc = 0 if C.stride(0) == N else C.stride(0)
    return Nvfp4Problem(M, N, K, sf_layout, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                        C.data_ptr(), ldc, 0)


def prepack_scales(sf_rowmajor, K: int, out=None, stream=None):
    """Blocked copy of a row-major uint8 [rows, K/16] CUDA tensor (a new tensor unless `out` is given)."""
    import torch
    rows = sf_rowmajor.shape[0]
    if out is None:
        out = torch.empty(max(1, nvfp4_prepacked_scale_bytes(rows, K)), dtype=torch.uint8, device=sf_rowmajor.device)
    nvfp4_prepack_scales(sf_rowmajor.data_ptr(), rows, K, out.data_ptr(), stream)
    return out


def nvfp4_grouped_gemm_noalloc(probs: Sequence[Nvfp4Problem], stream=None, check: bool = True) -> int:
    """The grouped GEMM without any device allocation: its problem table lives in a
    fixed 256 KB array inside the library (see the C header for the limits)."""
    arr = (Nvfp4Problem * max(1, len(probs)))(*probs)
    rc = _get().nvfp4_grouped_gemm_noalloc(len(probs), arr, _stream_handle(stream))
    return _check(rc, "nvfp4_grouped_gemm_noalloc") if check else rc


def nvfp4_noalloc_status(stream=None) -> Tuple[int, List[int]]:
    """(status, [code, role, item, stage]) of the no-allocation kernel's error words; reading clears them."""
    st = ctypes.c_int(0)
    detail = (ctypes.c_int32 * 4)()
    _check(_get().nvfp4_noalloc_status(_stream_handle(stream), ctypes.byref(st), detail), "nvfp4_noalloc_status")
    return st.value, list(detail)
