"""Parity of the swapped-operand kernels (swap-AB: rows of B on the MMA's M side, the group's
rows of A on its N side, stream-K over the SMs) with the CPU oracle, through the C ABI: the
single-CTA kernel (128 rows of B, up to 2 x 128 rows of A per item) and the CTA-pair kernel
(256 rows of B, up to 256 rows of A).

Bars, as for the other kernels: every output within |C_gpu - C_oracle| <= 1e-3 * S + 1 ulp16,
every output written, no store outside C, and the same bits on a repeated launch (split
tiles add their fp32 partials in K order whichever segment finishes last).
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity import assert_within_bound
import block_scaled_fp4_persistent_gb300 as nv
from gpu_util import DeviceGroup, run

pytestmark = pytest.mark.gpu

# NVFP4_OPT_CTA_PAIR values that select the swapped-operand kernels, and their names
KINDS = {3: "nvfp4_swapab_gemm_kernel<5>", 4: "nvfp4_swapab_pair_kernel<5>"}


@pytest.fixture(autouse=True, params=sorted(KINDS), ids=["single", "pair"])
def kind(request):
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, request.param)
    yield request.param
    for opt, val in [(nv.NVFP4_OPT_CTA_PAIR, 0), (nv.NVFP4_OPT_SPLIT_TAIL, 1), (nv.NVFP4_OPT_MAX_CTAS, 0),
                     (nv.NVFP4_OPT_SF_DIRECT, 1), (nv.NVFP4_OPT_PDL, 0)]:
        nv.nvfp4_set_option(opt, val)


def check_full(groups, dgroups, what):
    for i, ((c_ref, s_ref), d) in enumerate(zip(oracle.grouped_gemm(groups), dgroups)):
        got = d.result()
        assert not np.isnan(got).any(), f"{what} group {i}: unwritten outputs"
        assert_within_bound(got, c_ref, s_ref, f"{what} group {i}")
        assert d.guards_intact(), f"{what} group {i}: store outside C"


def rerun_same_bits(dgroups, what):
    first = [x.result().copy() for x in dgroups]
    for x in dgroups:
        x.reset()
    run(dgroups)
    for i, (f, x) in enumerate(zip(first, dgroups)):
        assert np.array_equal(f.view(np.uint16), x.result().view(np.uint16)), f"{what} group {i}: bits changed"


# M across the token-tile edges (16, 128, 256: one or two token tiles per item, a second
# item past 256), N across the B-tile edge, K with partial and whole last stages.
EDGES = dict(seed=301, Ms=[1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 300, 513],
             Ns=[8, 120, 128, 136, 264, 16, 72, 512, 8, 128, 200, 40],
             Ks=[64, 192, 256, 320, 1024, 64, 2304, 512, 128, 768, 256, 448])


@pytest.mark.parametrize("layout", [nv.NVFP4_SF_PREPACKED, nv.NVFP4_SF_ROWMAJOR])
def test_edges_of_the_token_and_weight_tiles(layout, kind):
    groups = gen.make_problem_set(EDGES["seed"], EDGES["Ms"], EDGES["Ns"], EDGES["Ks"])
    d = [DeviceGroup(g, layout) for g in groups]
    run(d)
    assert nv.nvfp4_last_kernel() == KINDS[kind]
    check_full(groups, d, f"swap-AB edges layout={layout}")
    rerun_same_bits(d, "swap-AB edges")


def test_row_major_scales_in_the_kernel_give_the_prepacked_bits():
    groups = gen.make_problem_set(302, [1, 40, 129, 248, 300], [8, 136, 264, 128, 72], [256, 512, 1024, 2304, 256])
    rm = [DeviceGroup(g, nv.NVFP4_SF_ROWMAJOR) for g in groups]
    run(rm)
    assert nv.nvfp4_last_launches() == 1
    check_full(groups, rm, "swap-AB row-major in the kernel")
    pre = [DeviceGroup(g) for g in groups]
    run(pre)
    for a, b in zip(rm, pre):
        assert np.array_equal(a.result().view(np.uint16), b.result().view(np.uint16))


@pytest.mark.parametrize("max_ctas", [0, 100, 37, 7, 1])
@pytest.mark.parametrize("split", [1, 0])
def test_stream_k_grids_match_oracle_and_are_deterministic(max_ctas, split):
    # Uniform K = 7168 (28 stages), groups with one, two and three token tiles: grids of
    # 152, 100, 37 and 7 CTAs cut items along K (stream-K) where it pays; 1 CTA runs every
    # item whole. With split 0 every item is whole.
    groups = gen.make_problem_set(303, [80, 176, 300, 64], [1024, 512, 384, 1024], [7168] * 4)
    nv.nvfp4_set_option(nv.NVFP4_OPT_MAX_CTAS, max_ctas)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, split)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, f"stream-K max_ctas={max_ctas} split={split}")
    rerun_same_bits(d, f"stream-K max_ctas={max_ctas} split={split}")


def test_many_groups():
    rng = np.random.default_rng(4)
    Ms = [int(m) for m in rng.integers(1, 400, 40)]
    Ns = [int(n) * 8 for n in rng.integers(1, 48, 40)]
    Ks = [int(k) * 64 for k in rng.integers(1, 24, 40)]
    groups = gen.make_problem_set(304, Ms, Ns, Ks)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, "swap-AB 40 groups")


def test_empty_groups_and_k0():
    groups = gen.make_problem_set(305, [0, 64, 3, 0, 130], [64, 0, 16, 8, 256], [256, 256, 0, 0, 128])
    d = [DeviceGroup(g) for g in groups]
    run(d)
    assert np.all(d[2].result() == 0)
    check_full([groups[4]], [d[4]], "swap-AB after empties")


def test_structured_closed_form():
    # all elements 1.0, scales 0.5 and 2: C = K exactly, in every row and column
    class G:
        pass
    groups = []
    for M, N, K in [(130, 200, 2048), (5, 8, 64), (257, 136, 7168)]:
        g = G()
        g.M, g.N, g.K = M, N, K
        g.A = np.full((M, K // 2), 0x22, np.uint8)
        g.B = np.full((N, K // 2), 0x22, np.uint8)
        g.SFA = np.full((M, K // 16), 0x30, np.uint8)
        g.SFB = np.full((N, K // 16), 0x40, np.uint8)
        groups.append(g)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    for g, dg in zip(groups, d):
        assert np.all(dg.result().astype(np.float64) == g.K)


def test_dependent_launch_and_two_calls_into_one_c():
    nv.nvfp4_set_option(nv.NVFP4_OPT_PDL, 1)
    first = gen.make_problem_set(306, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    second = gen.make_problem_set(307, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    d1 = [DeviceGroup(g) for g in first]
    d2 = [DeviceGroup(g) for g in second]
    probs2 = []
    for x1, x2 in zip(d1, d2):
        p = x2.problem()
        p.C = x1.problem().C
        probs2.append(p)
    nv.nvfp4_grouped_gemm([x.problem() for x in d1])
    nv.nvfp4_grouped_gemm(probs2)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status()[0] == 0
    check_full(second, d1, "swap-AB with PDL, two calls into one C")


def test_cuda_graph_capture_and_replay():
    groups = gen.make_problem_set(308, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    d = [DeviceGroup(g) for g in groups]
    probs = [x.problem() for x in d]
    run(d)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        nv.nvfp4_grouped_gemm(probs, s.cuda_stream)
    for _ in range(2):
        for x in d:
            x.reset()
        graph.replay()
        torch.cuda.synchronize()
        check_full(groups, d, "swap-AB graph replay")


CASES = 24


@pytest.mark.parametrize("case", range(CASES))
def test_random_problem_sets_match_oracle(case):
    rng = np.random.default_rng(3000 + case)
    g = int(rng.integers(1, 6))
    K = int(rng.integers(1, 40)) * 64
    Ms = [int(rng.integers(1, 400)) for _ in range(g)]
    Ns = [int(rng.integers(1, 65)) * 8 for _ in range(g)]
    Ks = [K if rng.random() < 0.8 else int(rng.integers(1, 40)) * 64 for _ in range(g)]
    layout = nv.NVFP4_SF_ROWMAJOR if rng.random() < 0.5 else nv.NVFP4_SF_PREPACKED
    split = int(rng.integers(0, 2))
    max_ctas = [0, 0, 5, 19, 64][int(rng.integers(0, 5))]
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, split)
    nv.nvfp4_set_option(nv.NVFP4_OPT_MAX_CTAS, max_ctas)
    groups = gen.make_problem_set(6000 + case, Ms, Ns, Ks)
    d = [DeviceGroup(g, layout) for g in groups]
    run(d)
    check_full(groups, d, f"case {case}: M={Ms} N={Ns} K={Ks} layout={layout} split={split} max_ctas={max_ctas}")
