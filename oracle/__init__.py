"""CPU oracle for the grouped NVFP4 block-scaled GEMM. TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this module. The CUDA library shares no code with it.

The arithmetic lives in ``nvfp4_oracle.c``, which cites the passages it
follows. This wrapper compiles that file with gcc and passes numpy arrays
to it:

* ``grouped_gemm``: every output of every group, plus the per-output
  magnitude sum that the tolerance needs;
* ``gemm_entries``: chosen outputs of one group, one by one, so that
  full-size workloads can be checked by sampling;
* ``blocked_scales``: the 128 x 4 blocked scale layout;
* ``e2m1``, ``e4m3``, ``fp16_rne``: the element decoders and the rounding.

Parity status: every function here is pinned by tests in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_nvfp4.so")
_lock = threading.Lock()
_lib = None


class OracleProblem(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("SFA", ctypes.c_void_p), ("SFB", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("S", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle_nvfp4.so`` next to its source."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_e2m1.restype = ctypes.c_double
        lib.oracle_e2m1.argtypes = [ctypes.c_uint]
        lib.oracle_e4m3.restype = ctypes.c_double
        lib.oracle_e4m3.argtypes = [ctypes.c_uint]
        lib.oracle_fp16_rne.restype = ctypes.c_uint16
        lib.oracle_fp16_rne.argtypes = [ctypes.c_double]
        lib.oracle_grouped_gemm.restype = ctypes.c_int
        lib.oracle_grouped_gemm.argtypes = [ctypes.c_int, ctypes.POINTER(OracleProblem), ctypes.c_int]
        lib.oracle_gemm_entries.restype = ctypes.c_int
        lib.oracle_gemm_entries.argtypes = [ctypes.POINTER(OracleProblem), ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_blocked_scale_bytes.restype = ctypes.c_size_t
        lib.oracle_blocked_scale_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.oracle_blocked_scales.restype = ctypes.c_int
        lib.oracle_blocked_scales.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        _lib = lib
        return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def e2m1(code: int) -> float:
    return _load().oracle_e2m1(code)


def e4m3(byte: int) -> float:
    return _load().oracle_e4m3(byte)


def fp16_rne(x: float) -> int:
    """The oracle's double -> fp16 rounding, as a 16-bit pattern."""
    return int(_load().oracle_fp16_rne(float(x)))


def _u8(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8, got {a.dtype}")
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data if a.size else 0


def _problem(M, N, K, A, B, SFA, SFB, C=None, S=None) -> Tuple[OracleProblem, list]:
    A, B, SFA, SFB = _u8(A), _u8(B), _u8(SFA), _u8(SFB)
    if A.size != M * (K // 2) or B.size != N * (K // 2) or SFA.size != M * (K // 16) or SFB.size != N * (K // 16):
        raise ValueError("operand sizes do not match M, N, K")
    p = OracleProblem(M, N, K, _ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB),
                      _ptr(C) if C is not None else 0, _ptr(S) if S is not None else 0)
    return p, [A, B, SFA, SFB, C, S]


def grouped_gemm(groups: Sequence, nthreads: Optional[int] = None,
                 want_abs: bool = True) -> List[Tuple[np.ndarray, Optional[np.ndarray]]]:
    """Every output of every group.

    ``groups`` holds objects with fields M, N, K, A, B, SFA and SFB, in the
    layouts of ``gen.GroupInputs``. Returns one (C, S) pair per group:
    C is float16 [M, N] and S is float64 [M, N], or None if want_abs is False.
    """
    lib = _load()
    out, keep = [], []
    probs = (OracleProblem * max(1, len(groups)))()
    for i, gi in enumerate(groups):
        C = np.zeros((gi.M, gi.N), dtype=np.uint16)
        S = np.zeros((gi.M, gi.N), dtype=np.float64) if want_abs else None
        p, k = _problem(gi.M, gi.N, gi.K, gi.A, gi.B, gi.SFA, gi.SFB, C, S)
        probs[i] = p
        keep.append(k)
        out.append((C, S))
    rc = lib.oracle_grouped_gemm(len(groups), probs, nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_grouped_gemm failed ({rc})")
    return [(C.view(np.float16), S) for C, S in out]


def gemm_entries(gi, ms: Sequence[int], ns: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Outputs (ms[i], ns[i]) of one group: float16 values and float64 magnitude sums."""
    lib = _load()
    m = np.ascontiguousarray(ms, dtype=np.int32)
    n = np.ascontiguousarray(ns, dtype=np.int32)
    if m.shape != n.shape:
        raise ValueError("ms and ns differ in length")
    c = np.zeros(m.size, dtype=np.uint16)
    s = np.zeros(m.size, dtype=np.float64)
    p, keep = _problem(gi.M, gi.N, gi.K, gi.A, gi.B, gi.SFA, gi.SFB)
    rc = lib.oracle_gemm_entries(ctypes.byref(p), m.size, _ptr(m), _ptr(n), _ptr(c), _ptr(s))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_entries failed ({rc})")
    return c.view(np.float16), s


def blocked_scale_bytes(rows: int, cols: int) -> int:
    return int(_load().oracle_blocked_scale_bytes(rows, cols))


def blocked_scales(sf: np.ndarray) -> np.ndarray:
    """The 128 x 4 blocked layout of a row-major [rows, cols] scale matrix."""
    sf = _u8(sf)
    rows, cols = sf.shape
    out = np.zeros(blocked_scale_bytes(rows, cols), dtype=np.uint8)
    rc = _load().oracle_blocked_scales(_ptr(sf), rows, cols, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_blocked_scales failed")
    return out
