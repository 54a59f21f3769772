"""The acceptance bound that compares the CUDA path's outputs with the oracle's.

After the fp16 rounding, each GPU output must satisfy

    |C_gpu - C_oracle| <= 1e-3 * S + ulp16(C_oracle)

where S = sum_k |a * sa * b * sb| is the oracle's magnitude sum for that
output. ulp16(x) is the fp16 spacing at |x|: 2^(floor(log2|x|) - 10) for
normal values and 2^-24 for subnormals and zero.

Why this bound. The tensor core adds fp32 partial sums in an order of its own,
so several fp16 results are correct. fp32 addition errs by at most about
K * 2^-24 * S. That is below 1e-3 * S for every K here (K <= 2^14). The final
rounding to fp16 adds at most half an ulp, and a partial sum that lands near
a tie can move the result by one more ulp. An output that is wrong for any
other reason (a dropped block, a wrong scale, a swapped nibble) is off by
much more than this.

Signed zeros compare equal. Equal infinities compare equal.
"""
import numpy as np

REL = 1e-3


def ulp16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x.astype(np.float64))
    out = np.full(a.shape, 2.0 ** -24)
    normal = a >= 2.0 ** -14
    out[normal] = np.exp2(np.floor(np.log2(a[normal])) - 10)
    return out


def violations(c_gpu: np.ndarray, c_ref: np.ndarray, s_ref: np.ndarray):
    """Boolean mask of outputs outside the bound."""
    g = np.asarray(c_gpu, dtype=np.float16).astype(np.float64)
    r = np.asarray(c_ref, dtype=np.float16).astype(np.float64)
    s = np.asarray(s_ref, dtype=np.float64)
    both_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):
        bad = ~(np.abs(g - r) <= REL * s + ulp16(r))
    return bad & ~both_inf


def assert_within_bound(c_gpu, c_ref, s_ref, what=""):
    bad = violations(c_gpu, c_ref, s_ref)
    if bad.any():
        idx = np.argwhere(bad)
        first = tuple(idx[0])
        g = np.asarray(c_gpu, dtype=np.float16)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside the bound; first at {first}: "
            f"gpu={float(g[first])} oracle={float(np.asarray(c_ref)[first])} S={float(np.asarray(s_ref)[first])}")
