"""Pins for the CPU oracle. Each one checks it against something other than itself.

Each pin is chosen so that a plausible mistake somewhere in the oracle fails
at least one of them:

* a wrong table entry or sign: the page's printed E2M1 table, plus E2M1
  decoded from its bit fields;
* a wrong E4M3 exponent or bias, or a broken subnormal or NaN: all 256 codes
  against torch's float8_e4m3fn conversion, a library routine;
* a wrong fp16 rounding: exhaustive comparison with numpy's float64->float16
  cast on every fp16 value, midpoint and boundary;
* swapped nibbles, a wrong scale index or a transposed operand: hand-worked
  1x1x16 and 2x2x32 cases;
* a dropped or doubled K block: the closed form C = K * sa * sb for all-ones
  inputs;
* anything else: brute force with exact rationals on tiny shapes, plus the
  sign, scale, transpose, permutation, split and zero-padding invariants.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- helpers ---

class G:
    """A group built by hand from row-major arrays."""

    def __init__(self, A, B, SFA, SFB):
        self.A = np.ascontiguousarray(A, dtype=np.uint8)
        self.B = np.ascontiguousarray(B, dtype=np.uint8)
        self.SFA = np.ascontiguousarray(SFA, dtype=np.uint8)
        self.SFB = np.ascontiguousarray(SFB, dtype=np.uint8)
        self.M, self.N = self.A.shape[0], self.B.shape[0]
        self.K = self.A.shape[1] * 2


def run1(g):
    (c, s), = oracle.grouped_gemm([g], nthreads=2)
    return c, s


def bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def e2m1_from_fields(code: int) -> Fraction:
    """E2M1 from its bit fields: sign bit 3, a 2-bit exponent with bias 1, and
    1 mantissa bit. Exponent 0 is subnormal (m * 1/2)."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -v if s else v


_E4M3_TORCH = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_force(g) -> np.ndarray:
    """Exact rational sum, cast once with numpy's float16 conversion. Shares no code with the oracle."""
    M, N, K = g.M, g.N, g.K

    def vals(P, SF, r):
        out = []
        for k in range(K):
            byte = int(P[r, k // 2])
            code = (byte >> 4) if (k % 2) else (byte & 0xF)
            out.append(e2m1_from_fields(code) * Fraction(float(_E4M3_TORCH[int(SF[r, k // 16])])))
        return out

    C = np.zeros((M, N), dtype=np.float16)
    arows = [vals(g.A, g.SFA, m) for m in range(M)]
    brows = [vals(g.B, g.SFB, n) for n in range(N)]
    for m in range(M):
        for n in range(N):
            exact = sum((a * b for a, b in zip(arows[m], brows[n])), Fraction(0))
            C[m, n] = np.float16(float(exact))  # exact in double (< 53 bits), then one rounding
    return C


# -------------------------------------------------------- element decoders ---

def test_e2m1_matches_page_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_table.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s), float(val_s)
        got = oracle.e2m1(code)
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_e2m1_matches_bit_field_definition():
    for code in range(16):
        assert Fraction(oracle.e2m1(code)) == e2m1_from_fields(code), code


def test_e4m3_all_codes_match_torch():
    for b in range(256):
        got, ref = oracle.e4m3(b), float(_E4M3_TORCH[b])
        if np.isnan(ref):
            assert np.isnan(got), hex(b)
        else:
            assert got == ref and np.signbit(got) == np.signbit(ref), (hex(b), got, ref)


def test_e4m3_spot_values():
    assert oracle.e4m3(0x01) == 2.0 ** -9
    assert oracle.e4m3(0x08) == 2.0 ** -6
    assert oracle.e4m3(0x38) == 1.0
    assert oracle.e4m3(0x20) == 0.125 and oracle.e4m3(0x40) == 2.0
    assert oracle.e4m3(0x7E) == 448.0
    assert np.isnan(oracle.e4m3(0x7F)) and np.isnan(oracle.e4m3(0xFF))
    z = oracle.e4m3(0x80)
    assert z == 0.0 and np.signbit(z)


# ------------------------------------------------------------ fp16 rounding ---

def _fp16_probe_points():
    h = np.arange(0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)  # all finite non-negative
    nxt = np.append(h[1:], 65536.0)  # next value up (65536 = the 'next' after max for rounding purposes)
    mids = (h + nxt) / 2
    pts = [h, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf), np.nextafter(h, 0), np.nextafter(h, np.inf)]
    extra = np.array([0.0, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26, 65504.0, 65519.999, 65520.0, 65536.0, 1e9,
                      2.0 ** -14 - 2.0 ** -25, 2.0 ** -14 - 2.0 ** -26])
    allp = np.concatenate(pts + [extra])
    return np.concatenate([allp, -allp])


def test_fp16_rne_matches_numpy_everywhere():
    lib = oracle._load()
    pts = _fp16_probe_points()
    got = np.array([lib.oracle_fp16_rne(float(x)) for x in pts], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = pts.astype(np.float16).view(np.uint16)
    mism = np.nonzero(got != ref)[0]
    assert mism.size == 0, [(pts[i], hex(got[i]), hex(ref[i])) for i in mism[:5]]


def test_fp16_rne_random_doubles():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000))
    lib = oracle._load()
    got = np.array([lib.oracle_fp16_rne(float(v)) for v in x], dtype=np.uint16)
    with np.errstate(over="ignore"):
        assert np.array_equal(got, x.astype(np.float16).view(np.uint16))
    assert oracle.fp16_rne(float("nan")) & 0x7C00 == 0x7C00


# -------------------------------------------------------- hand-worked cases ---

def test_hand_worked_1x1x16():
    # A = B = codes 0..15 in k order (bytes 0x10 0x32 .. 0xFE), SFA = 0x38 (1.0), SFB = 0x30 (0.5).
    # sum_k a_k^2 = 2 * (0 + .25 + 1 + 2.25 + 4 + 9 + 16 + 36) = 137; times 1.0 * 0.5 = 68.5.
    row = np.array([[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]], dtype=np.uint8)
    c, s = run1(G(row, row, [[0x38]], [[0x30]]))
    assert c.shape == (1, 1) and float(c[0, 0]) == 68.5
    assert s[0, 0] == 68.5


def test_hand_worked_2x2x32():
    # A row 0: all 1.0 (0x22), SFA [1, 2]; A row 1: k even +1, k odd -0.5 (0x92), SFA [1, 1].
    # B row 0: all 0.5 (0x11), SFB [1, .5]; B row 1: all 6 (0x77), SFB [.25, 1].
    # C00 = 16*1*1*.5*1 + 16*1*2*.5*.5 = 8 + 8 = 16
    # C01 = 16*1*1*6*.25 + 16*1*2*6*1 = 24 + 192 = 216
    # C10 = 8*(1-.5)*.5*1 + 8*(1-.5)*.5*.5 = 2 + 1 = 3
    # C11 = 8*(1-.5)*6*.25 + 8*(1-.5)*6*1 = 6 + 24 = 30
    A = np.array([[0x22] * 16, [0x92] * 16], dtype=np.uint8)
    B = np.array([[0x11] * 16, [0x77] * 16], dtype=np.uint8)
    SFA = np.array([[0x38, 0x40], [0x38, 0x38]], dtype=np.uint8)
    SFB = np.array([[0x38, 0x30], [0x28, 0x38]], dtype=np.uint8)
    c, _ = run1(G(A, B, SFA, SFB))
    assert c.astype(np.float64).tolist() == [[16.0, 216.0], [3.0, 30.0]]


@pytest.mark.parametrize("K", [16, 64, 512, 1536, 2048, 4096, 7168])
@pytest.mark.parametrize("sa,sb,scale", [(0x38, 0x38, 1.0), (0x30, 0x40, 1.0), (0x28, 0x3C, 0.375)])
def test_closed_form_all_ones(K, sa, sb, scale):
    # every element is 1.0 (byte 0x22), so C = K * sa * sb exactly (all of these fit fp16 exactly)
    M, N = 3, 5
    A = np.full((M, K // 2), 0x22, np.uint8)
    B = np.full((N, K // 2), 0x22, np.uint8)
    c, s = run1(G(A, B, np.full((M, K // 16), sa, np.uint8), np.full((N, K // 16), sb, np.uint8)))
    assert np.all(c.astype(np.float64) == K * scale)
    assert np.all(s == K * scale)


# ----------------------------------------------------------- brute force ---

@pytest.mark.parametrize("K", [16, 32, 64, 256])
@pytest.mark.parametrize("wide_scales", [False, True])
def test_brute_force_tiny(K, wide_scales):
    rng = np.random.default_rng(1000 + K + 7 * wide_scales)
    M, N = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    A = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    if wide_scales:  # every finite non-negative code, subnormals included
        codes = np.arange(0x00, 0x7F, dtype=np.uint8)
        SFA, SFB = rng.choice(codes, (M, K // 16)), rng.choice(codes, (N, K // 16))
    else:
        SFA = rng.integers(0x20, 0x41, (M, K // 16), dtype=np.uint8)
        SFB = rng.integers(0x20, 0x41, (N, K // 16), dtype=np.uint8)
    g = G(A, B, SFA, SFB)
    c, _ = run1(g)
    ref = brute_force(g)
    assert np.array_equal(np.where(c == 0, 0, bits(c)), np.where(ref == 0, 0, bits(ref)))


def test_brute_force_generated_small():
    groups = gen.make_problem_set(5, [3, 2], [2, 4], [64, 32])
    outs = oracle.grouped_gemm(groups, nthreads=3)
    for g, (c, _) in zip(groups, outs):
        ref = brute_force(g)
        assert np.array_equal(np.where(c == 0, 0, bits(c)), np.where(ref == 0, 0, bits(ref)))


# -------------------------------------------------------------- invariants ---

def _gen_small(seed=3, M=9, N=12, K=128):
    return gen.make_group(seed, 0, M, N, K)


def _eq(a, b):
    a, b = np.asarray(a, np.float16), np.asarray(b, np.float16)
    return np.array_equal(np.where(a == 0, 0, bits(a)), np.where(b == 0, 0, bits(b)))


def test_invariant_sign():
    g = _gen_small()
    c, _ = run1(g)
    neg = G(g.A ^ 0x88, g.B, g.SFA, g.SFB)
    cn, _ = run1(neg)
    assert _eq(cn, -c)


def test_invariant_scale_doubling():
    g = _gen_small()  # scale codes 0x20..0x40 are normal; +8 adds one to the exponent
    c, _ = run1(g)
    c2, _ = run1(G(g.A, g.B, g.SFA + 8, g.SFB))
    assert _eq(c2, (c.astype(np.float64) * 2).astype(np.float16))


def test_invariant_transpose():
    g = _gen_small()
    c, _ = run1(g)
    ct, _ = run1(G(g.B, g.A, g.SFB, g.SFA))
    assert _eq(ct, c.T)


def test_invariant_group_permutation_and_split():
    groups = gen.make_problem_set(11, [5, 7, 4], [8, 16, 24], [64, 96, 32])
    outs = oracle.grouped_gemm(groups, nthreads=2)
    perm = [2, 0, 1]
    outs_p = oracle.grouped_gemm([groups[i] for i in perm], nthreads=2)
    for j, i in enumerate(perm):
        assert _eq(outs_p[j][0], outs[i][0])
    # split group 1 along M (rows 0..2 / 3..6) and along N (cols 0..9 / 10..15)
    g = groups[1]
    top = G(g.A[:3], g.B, g.SFA[:3], g.SFB)
    bot = G(g.A[3:], g.B, g.SFA[3:], g.SFB)
    left = G(g.A, g.B[:10], g.SFA, g.SFB[:10])
    right = G(g.A, g.B[10:], g.SFA, g.SFB[10:])
    full = outs[1][0]
    assert _eq(run1(top)[0], full[:3]) and _eq(run1(bot)[0], full[3:])
    assert _eq(run1(left)[0], full[:, :10]) and _eq(run1(right)[0], full[:, 10:])


def test_invariant_zero_padding_of_k():
    g = _gen_small(K=96)
    c, s = run1(g)
    pad = lambda P, n: np.concatenate([P, np.zeros((P.shape[0], n), np.uint8)], axis=1)
    # 64 more K: 32 more zero bytes per row and 4 more scale blocks (nonzero scales, zero data)
    gp = G(pad(g.A, 32), pad(g.B, 32), np.concatenate([g.SFA, np.full((g.M, 4), 0x38, np.uint8)], 1),
           np.concatenate([g.SFB, np.full((g.N, 4), 0x40, np.uint8)], 1))
    cp, sp = run1(gp)
    assert _eq(cp, c) and np.array_equal(sp, s)


# ------------------------------------------------------ sampled entries ---

def test_entries_equal_full_computation():
    g = gen.make_group(21, 0, 37, 48, 256)
    (c, s), = oracle.grouped_gemm([g], nthreads=4)
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, g.M, 200), rng.integers(0, g.N, 200)
    ce, se = oracle.gemm_entries(g, ms, ns)
    assert np.array_equal(bits(ce), bits(c[ms, ns])) and np.array_equal(se, s[ms, ns])


def test_empty_and_degenerate_shapes():
    g0 = gen.make_group(1, 0, 0, 8, 64)
    g1 = gen.make_group(1, 1, 4, 0, 64)
    g2 = G(np.zeros((3, 0), np.uint8), np.zeros((5, 0), np.uint8), np.zeros((3, 0), np.uint8), np.zeros((5, 0), np.uint8))
    outs = oracle.grouped_gemm([g0, g1, g2], nthreads=2)
    assert outs[0][0].shape == (0, 8) and outs[1][0].shape == (4, 0)
    assert outs[2][0].shape == (3, 5) and np.all(outs[2][0] == 0)  # K = 0: the empty sum


# ------------------------------------------------------ blocked scale layout ---

@pytest.mark.parametrize("rows,cols", [(1, 4), (128, 4), (129, 8), (300, 28), (40, 128), (256, 448), (7, 6)])
def test_blocked_layout_element_positions(rows, cols):
    # Pinned by the element -> byte map that the kernels on page 1 and page 3 index with:
    # the 512-byte block of (row tile r/128, column block c/4) sits at ((r/128) * ceil(cols/4) + c/4) * 512,
    # and inside it the page-4 atom strides ((16,4),(0,1)) put (r, c) at (r%32)*16 + ((r%128)/32)*4 + c%4.
    rng = np.random.default_rng(rows * 1000 + cols)
    sf = rng.integers(1, 256, (rows, cols), dtype=np.uint8)  # nonzero, so padding is visible
    out = oracle.blocked_scales(sf)
    ncb = (cols + 3) // 4
    assert out.size == ((rows + 127) // 128) * 128 * ncb * 4
    seen = np.zeros(out.size, bool)
    for r in range(rows):
        for c in range(cols):
            off = ((r // 128) * ncb + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
            assert out[off] == sf[r, c]
            seen[off] = True
    assert np.all(out[~seen] == 0)
