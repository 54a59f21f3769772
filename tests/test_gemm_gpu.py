"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Bars:
 * scale prepack: byte-for-byte identical to the oracle's blocked layout;
 * GEMM: every compared output within |C_gpu - C_oracle| <= 1e-3 * S + 1 ulp16;
 * no store outside C (4 KB canary bands on both sides) and no output left unwritten;
 * results independent of the pipeline depth and of the number of CTAs, bit for bit.
Every test compares every output, the full-size workloads included (in the launch
configuration the benchmark uses, and in the others).
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity import assert_within_bound
import block_scaled_fp4_persistent_gb300 as nv
from gpu_util import DeviceGroup, run, workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for opt, val in [(nv.NVFP4_OPT_STAGES, 0), (nv.NVFP4_OPT_MAX_CTAS, 0), (nv.NVFP4_OPT_BLOCK_N, 0),
                     (nv.NVFP4_OPT_FAULT_SKIP_LOAD, -1), (nv.NVFP4_OPT_WAIT_TIMEOUT_US, 2000000),
                     (nv.NVFP4_OPT_SPLIT_TAIL, 1), (nv.NVFP4_OPT_CTA_PAIR, 0), (nv.NVFP4_OPT_SF_DIRECT, 1),
                     (nv.NVFP4_OPT_PDL, 0), (nv.NVFP4_OPT_M_FUSION, 1)]:
        nv.nvfp4_set_option(opt, val)


def check_full(groups, dgroups, what):
    ref = oracle.grouped_gemm(groups)
    for i, ((c_ref, s_ref), d) in enumerate(zip(ref, dgroups)):
        got = d.result()
        assert not np.isnan(got).any(), f"{what} group {i}: unwritten outputs"
        assert_within_bound(got, c_ref, s_ref, f"{what} group {i}")
        assert d.guards_intact(), f"{what} group {i}: store outside C"


# ------------------------------------------------------------------ prepack --

@pytest.mark.parametrize("rows,K", [(1, 64), (40, 2048), (128, 256), (129, 320), (300, 1024), (248, 7168),
                                    (7, 48), (4096, 1536)])
def test_prepack_bitwise(rows, K):
    rng = np.random.default_rng(rows + K)
    sf = rng.integers(0, 256, (rows, K // 16), dtype=np.uint8)
    out = nv.prepack_scales(torch.from_numpy(sf).cuda(), K)
    torch.cuda.synchronize()
    ref = oracle.blocked_scales(sf)
    assert np.array_equal(out.cpu().numpy()[:ref.size], ref)


def test_prepack_batch_mixed_operands():
    # one launch over operands of both load paths: 16-byte rows (K % 256 == 0; 28, 3 and
    # 1 sixteen-column pieces per row) and byte rows (K / 16 = 3, 20, 25); each output
    # byte-for-byte the oracle's, the 64 guard bytes after each untouched
    shapes = [(300, 7168), (129, 768), (7, 48), (1000, 320), (128, 256), (257, 400), (40, 2048)]
    rng = np.random.default_rng(77)
    srcs, dsts, refs, guard = [], [], [], 64
    for rows, K in shapes:
        sf = rng.integers(0, 256, (rows, K // 16), dtype=np.uint8)
        srcs.append(torch.from_numpy(sf).cuda())
        refs.append(oracle.blocked_scales(sf))
        dsts.append(torch.full((nv.nvfp4_prepacked_scale_bytes(rows, K) + guard,), 0xEE, dtype=torch.uint8,
                               device="cuda"))
    nv.nvfp4_prepack_scales_batch([s.data_ptr() for s in srcs], [r for r, _ in shapes], [k for _, k in shapes],
                                  [d.data_ptr() for d in dsts])
    torch.cuda.synchronize()
    for (rows, K), d, ref in zip(shapes, dsts, refs):
        got = d.cpu().numpy()
        assert got.size - guard == ref.size
        assert np.array_equal(got[:ref.size], ref), f"rows={rows} K={K}"
        assert np.all(got[ref.size:] == 0xEE), f"rows={rows} K={K}: store past the blocked layout"


# ------------------------------------------------------------ small, full ---

def test_decode_sized_sets_take_the_swapped_kernel():
    # every group at most 32 rows of A: the automatic choice is the swapped-operand kernel
    groups = gen.make_problem_set(11, [8, 16, 4, 32, 1, 3], [4096, 512, 1024, 136, 8, 264], [7168, 256, 1024, 2048, 64, 448])
    d = [DeviceGroup(g) for g in groups]
    run(d)
    assert nv.nvfp4_last_kernel() == "nvfp4_swapab_gemm_kernel<5>"
    check_full(groups, d, "decode-sized set")


def test_tiny_workload_every_output():
    groups = gen.make_workload("tiny_g2")
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, "tiny_g2")
    assert nv.nvfp4_last_kernel().startswith("nvfp4_grouped_gemm_kernel<")  # small sets: single CTAs


def test_last_kernel_names_the_variant_that_ran():
    groups = gen.make_problem_set(3, [130], [512], [256])
    for pair, name in [(1, "nvfp4_pair_gemm_kernel<5>"), (2, "nvfp4_grouped_gemm_kernel<128,5>")]:
        nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
        d = [DeviceGroup(g) for g in groups]
        run(d)
        assert nv.nvfp4_last_kernel() == name
        check_full(groups, d, name)


RAGGED = dict(seed=77, Ms=[1, 40, 127, 128, 129, 248, 300], Ns=[8, 120, 136, 512, 264, 128, 72],
              Ks=[64, 192, 256, 320, 1024, 512, 2304])


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("layout", [nv.NVFP4_SF_PREPACKED, nv.NVFP4_SF_ROWMAJOR])
def test_ragged_shapes_one_launch(layout, pair):
    # CTA pairs: M = 1..300 leaves the second CTA's rows partly or wholly past M, and
    # N = 8..264 leaves the second half of the B tile partly or wholly past N. With
    # row-major scales the groups with K % 256 == 0 read them in the kernel and the
    # others through the prepack kernel, in the same call.
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    groups = gen.make_problem_set(RAGGED["seed"], RAGGED["Ms"], RAGGED["Ns"], RAGGED["Ks"])
    d = [DeviceGroup(g, layout) for g in groups]
    run(d)
    assert nv.nvfp4_last_launches() == (2 if layout == nv.NVFP4_SF_ROWMAJOR else 1)
    check_full(groups, d, f"ragged layout={layout} pair={pair}")


# K % 256 == 0 throughout: every group reads its row-major scales in the kernel
DIRECT = dict(seed=78, Ms=[1, 40, 127, 129, 248, 300], Ns=[8, 136, 512, 264, 128, 72],
              Ks=[256, 512, 768, 1024, 2304, 256])


@pytest.mark.parametrize("pair,block_n", [(1, 0), (2, 0), (2, 256)])
def test_row_major_scales_read_in_the_kernel(pair, block_n):
    # one launch, and the same bits as prepacked scales and as the prepack route
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    nv.nvfp4_set_option(nv.NVFP4_OPT_BLOCK_N, block_n)
    groups = gen.make_problem_set(DIRECT["seed"], DIRECT["Ms"], DIRECT["Ns"], DIRECT["Ks"])
    d = [DeviceGroup(g, nv.NVFP4_SF_ROWMAJOR) for g in groups]
    run(d)
    assert nv.nvfp4_last_launches() == 1
    check_full(groups, d, f"row-major in the kernel pair={pair} block_n={block_n}")
    pre = [DeviceGroup(g) for g in groups]
    run(pre)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SF_DIRECT, 0)
    via = [DeviceGroup(g, nv.NVFP4_SF_ROWMAJOR) for g in groups]
    run(via)
    assert nv.nvfp4_last_launches() == 2
    for a, b, c in zip(d, pre, via):
        assert np.array_equal(a.result().view(np.uint16), b.result().view(np.uint16))
        assert np.array_equal(a.result().view(np.uint16), c.result().view(np.uint16))


@pytest.mark.parametrize("pair", [1, 2])
def test_dependent_launch_with_row_major_scales(pair):
    # row-major scales with K % 256 != 0 for some groups: a prepack launch, then the
    # dependent GEMM launch, which must wait for the prepacked scales
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    nv.nvfp4_set_option(nv.NVFP4_OPT_PDL, 1)
    groups = gen.make_problem_set(RAGGED["seed"] + 2, RAGGED["Ms"], RAGGED["Ns"], RAGGED["Ks"])
    d = [DeviceGroup(g, nv.NVFP4_SF_ROWMAJOR) for g in groups]
    run(d)
    assert nv.nvfp4_last_launches() == 2
    check_full(groups, d, f"dependent launch after the prepack, pair={pair}")


@pytest.mark.parametrize("pair", [1, 2])
def test_dependent_launch_waits_for_the_kernels_before_it(pair):
    # With programmatic dependent launch the GEMM may start while the kernel before
    # it finishes. Here that kernel writes the right inputs over wrong ones, and a
    # second GEMM call writes other results over the first call's C: the outputs
    # must be those of the right inputs and of the second call.
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    nv.nvfp4_set_option(nv.NVFP4_OPT_PDL, 1)
    first = gen.make_problem_set(81, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    second = gen.make_problem_set(82, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    d1 = [DeviceGroup(g) for g in first]
    d2 = [DeviceGroup(g) for g in second]
    right = [(x.A.clone(), x.B.clone()) for x in d1]
    for x in d1:
        x.A.fill_(0x77)
        x.B.fill_(0x77)
    zero = torch.zeros(1, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for x, (a, b) in zip(d1, right):
        torch.bitwise_or(a, zero, out=x.A)  # kernels, right before the GEMM in the same stream
        torch.bitwise_or(b, zero, out=x.B)
    nv.nvfp4_grouped_gemm([x.problem() for x in d1])
    torch.cuda.synchronize()
    check_full(first, d1, f"dependent launch, inputs written just before, pair={pair}")
    # two calls in a row into the same C: the second one's results must remain
    probs2 = []
    for x1, x2 in zip(d1, d2):
        p = x2.problem()
        p.C = x1.problem().C
        probs2.append(p)
    nv.nvfp4_grouped_gemm([x.problem() for x in d1])
    nv.nvfp4_grouped_gemm(probs2)
    torch.cuda.synchronize()
    status, detail = nv.nvfp4_device_status()
    assert status == 0, detail
    check_full(second, d1, f"dependent launch, two calls into one C, pair={pair}")


@pytest.mark.parametrize("pair", [1, 2])
def test_cuda_graph_capture_and_replay(pair):
    # Once a problem set's table is cached, a call records into a CUDA graph (no
    # allocation, no synchronisation inside) and the graph replays it.
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    groups = gen.make_problem_set(91, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    d = [DeviceGroup(g) for g in groups]
    probs = [x.problem() for x in d]
    run(d)  # warms the table cache
    for x in d:
        x.reset()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        nv.nvfp4_grouped_gemm(probs, s.cuda_stream)
    for _ in range(2):
        for x in d:
            x.reset()
        graph.replay()
        torch.cuda.synchronize()
        check_full(groups, d, f"graph replay pair={pair}")


def test_structured_closed_form():
    # all elements 1.0 with scales 0.5 and 2 (codes 0x30, 0x40): C = K exactly
    class G:
        pass
    groups = []
    for M, N, K in [(130, 200, 2048), (5, 8, 64)]:
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



@pytest.mark.parametrize("pair", [1, 2])
def test_large_closed_form_with_row_and_column_scales(pair):
    # Every element 1.0; A's scale depends on the row (0.5, 1, 2 for m % 3) and B's on the
    # column (0.25, 0.5, 1, 2 for n % 4), so C[m][n] = K * sa[m] * sb[n] exactly (a power of
    # two times K, at most 2^15). A 2048 x 8192 x 8192 group (hundreds of tiles, several
    # waves, the compute-heavy regime) and a ragged one; every output compared, which also
    # catches a row or column of outputs landing in the wrong place.
    class G:
        pass
    groups = []
    for M, N, K in [(2048, 8192, 8192), (300, 1000, 4096)]:
        g = G()
        g.M, g.N, g.K = M, N, K
        g.A = np.full((M, K // 2), 0x22, np.uint8)
        g.B = np.full((N, K // 2), 0x22, np.uint8)
        g.SFA = np.repeat(np.array([0x30, 0x38, 0x40], np.uint8)[np.arange(M) % 3][:, None], K // 16, axis=1)
        g.SFB = np.repeat(np.array([0x28, 0x30, 0x38, 0x40], np.uint8)[np.arange(N) % 4][:, None], K // 16, axis=1)
        groups.append(g)
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    for g, dg in zip(groups, d):
        sa = np.array([0.5, 1.0, 2.0])[np.arange(g.M) % 3]
        sb = np.array([0.25, 0.5, 1.0, 2.0])[np.arange(g.N) % 4]
        expect = g.K * sa[:, None] * sb[None, :]
        got = dg.result().astype(np.float64)
        bad = np.argwhere(got != expect)
        assert bad.size == 0, f"kind {pair} M={g.M}: {len(bad)} outputs wrong, first at {tuple(bad[0])}"
        assert dg.guards_intact()


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("stages", [2, 0])
@pytest.mark.parametrize("max_ctas", [1, 3, 0])
def test_tile_width_depth_and_grid_do_not_change_results(block_n, stages, max_ctas):
    groups = gen.make_problem_set(5, [200, 64, 129], [384, 256, 136], [1536, 512, 768])
    nv.nvfp4_set_option(nv.NVFP4_OPT_BLOCK_N, block_n)
    base = [DeviceGroup(g) for g in groups]
    run(base)
    if (stages, max_ctas) == (0, 0):
        check_full(groups, base, f"block_n={block_n}")
    nv.nvfp4_set_option(nv.NVFP4_OPT_STAGES, stages)
    nv.nvfp4_set_option(nv.NVFP4_OPT_MAX_CTAS, max_ctas)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    for a, b in zip(base, d):
        assert np.array_equal(a.result().view(np.uint16), b.result().view(np.uint16))
        assert b.guards_intact()


@pytest.mark.parametrize("block_n", [128, 256])
def test_ragged_shapes_both_tile_widths(block_n):
    nv.nvfp4_set_option(nv.NVFP4_OPT_BLOCK_N, block_n)
    groups = gen.make_problem_set(RAGGED["seed"] + 1, RAGGED["Ms"], RAGGED["Ns"], RAGGED["Ks"])
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, f"ragged block_n={block_n}")


# --------------------------------------------------------------- edge cases ---

def test_edge_cases_empty_groups_and_k0():
    groups = gen.make_problem_set(9, [0, 64, 3, 0, 130], [64, 0, 16, 8, 256], [256, 256, 0, 0, 128])
    d = [DeviceGroup(g) for g in groups]
    run(d)
    assert np.all(d[2].result() == 0)  # K = 0: the empty sum
    assert d[2].guards_intact()
    check_full([groups[4]], [d[4]], "after empties")
    nv.nvfp4_grouped_gemm([])  # g = 0


def test_repeated_calls_and_table_cache():
    ga = gen.make_problem_set(13, [96, 160], [256, 128], [512, 256])
    gb = gen.make_problem_set(14, [33], [64], [1024])
    da = [DeviceGroup(g) for g in ga]
    db = [DeviceGroup(g) for g in gb]
    run(da)
    first = [x.result().copy() for x in da]
    run(db)
    for x in da:
        x.reset()
    run(da)  # table cache hit
    for f, x in zip(first, da):
        assert np.array_equal(f.view(np.uint16), x.result().view(np.uint16))
    check_full(gb, db, "second problem set")



def test_table_cache_churn_evicts_and_reuses_buffers():
    # 40 problem sets (distinct C buffers, so distinct tables), called round-robin three
    # times: past the cache's 32 tables every miss evicts one, whose pooled buffers go back
    # to the pool once the stream event recorded after their last launch completes, and are
    # handed to later tables. Every output of the last round against the oracle.
    sets = [gen.make_problem_set(600 + i, [64 + i], [128 + 8 * (i % 4)], [256]) for i in range(40)]
    devs = [[DeviceGroup(g) for g in s] for s in sets]
    for _ in range(3):
        for d in devs:
            for x in d:
                x.reset()
            nv.nvfp4_grouped_gemm([x.problem() for x in d])
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status()[0] == 0
    for i, (s, d) in enumerate(zip(sets, devs)):
        check_full(s, d, f"set {i}")



def test_release_then_reuse():
    # nvfp4_release frees every table, pooled buffer, workspace and the error word; the
    # next calls rebuild them (a kernel kind that splits, so a workspace exists too)
    ga = gen.make_problem_set(611, [130, 60, 200, 129], [2048, 1024, 1536, 520], [2048] * 4)
    nv.nvfp4_set_option(nv.NVFP4_OPT_MAX_CTAS, 70)  # a short last wave: split tiles, a workspace
    da = [DeviceGroup(g) for g in ga]
    run(da)
    first = [x.result().copy() for x in da]
    nv.nvfp4_release()
    nv.nvfp4_release()  # twice: nothing left to free
    for x in da:
        x.reset()
    run(da)
    for f, x in zip(first, da):
        assert np.array_equal(f.view(np.uint16), x.result().view(np.uint16))
    check_full(ga, da, "after release")
    assert nv.nvfp4_device_status()[0] == 0



@pytest.mark.parametrize("pair", [0, 1, 2, 3])
def test_150_groups_every_kernel_kind(pair):
    # groups 0-7 take their tensor maps from the launch parameters, the rest from the table
    # with an acquire fence (and only those below 64 are prefetched): 150 small groups,
    # ragged M and N, three K values, on every kernel kind
    rng = np.random.default_rng(150)
    Ms = [int(m) for m in rng.integers(1, 200, 150)]
    Ns = [int(n) * 8 for n in rng.integers(1, 40, 150)]
    Ks = [[256, 512, 1024][int(k)] for k in rng.integers(0, 3, 150)]
    groups = gen.make_problem_set(151, Ms, Ns, Ks)
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, f"150 groups, kind {pair}")


def test_many_groups():
    rng = np.random.default_rng(3)
    Ms = [int(m) for m in rng.integers(1, 300, 40)]
    Ns = [int(n) * 8 for n in rng.integers(1, 48, 40)]
    Ks = [int(k) * 64 for k in rng.integers(1, 12, 40)]
    groups = gen.make_problem_set(17, Ms, Ns, Ks)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, "40 groups")


def test_streams_are_respected():
    groups = gen.make_problem_set(21, [128, 64], [512, 256], [1024, 512])
    d = [DeviceGroup(g) for g in groups]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nv.nvfp4_grouped_gemm([x.problem() for x in d], s)
    s.synchronize()
    status, _ = nv.nvfp4_device_status(s)
    assert status == 0
    check_full(groups, d, "side stream")


def test_two_streams_at_once_with_split_tails():
    # Different problem sets on two streams, queued back to back without a sync: each has its own
    # table, split workspace and counters. Single CTAs on a grid small enough to split the tails.
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 2)
    nv.nvfp4_set_option(nv.NVFP4_OPT_MAX_CTAS, 70)
    sets = [gen.make_problem_set(23, [130, 60, 200, 129], [2048, 1024, 1536, 520], [2048] * 4),
            gen.make_problem_set(24, [100, 33, 250], [1536, 2048, 1024], [1024] * 3)]
    dev = [[DeviceGroup(g) for g in groups] for groups in sets]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):  # the first call of each set builds its table; later ones overlap
        for d, st in zip(dev, streams):
            with torch.cuda.stream(st):
                nv.nvfp4_grouped_gemm([x.problem() for x in d], st)
    torch.cuda.synchronize()
    for st in streams:
        status, detail = nv.nvfp4_device_status(st)
        assert status == 0, f"device status {status}: {detail}"
    for groups, d in zip(sets, dev):
        check_full(groups, d, "two streams")


# ------------------------------------------------------- full-size, every output ---

@pytest.mark.parametrize("pair,layout", [(0, nv.NVFP4_SF_PREPACKED), (1, nv.NVFP4_SF_ROWMAJOR),
                                         (2, nv.NVFP4_SF_PREPACKED), (2, nv.NVFP4_SF_ROWMAJOR),
                                         (3, nv.NVFP4_SF_PREPACKED), (3, nv.NVFP4_SF_ROWMAJOR),
                                         (4, nv.NVFP4_SF_PREPACKED), (4, nv.NVFP4_SF_ROWMAJOR)])
@pytest.mark.parametrize("name", ["g2_n4096_k1536", "g2_n3072_k4096", "moe_g8_n7168_k2048", "moe_g8_n4096_k7168"])
def test_full_size_workloads_every_output(name, pair, layout):
    # pair 0: the automatic choice with prepacked scales, the benchmark's launch
    # configuration; 1: CTA pairs; 2: single CTAs (which split the MoE sets' last
    # wave along K); 3 and 4: the swapped-operand kernels, single CTAs and CTA pairs
    # (stream-K). Row-major scales are read in the kernel (the e2e benchmark's route).
    # Every output is compared with the oracle's.
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, pair)
    groups = gen.make_workload(name)
    d = [DeviceGroup(g, layout) for g in groups]
    run(d)  # default options: the launch configuration of the benchmark
    for i, (x, (c_ref, s_ref)) in enumerate(zip(d, workload_reference(name))):
        got = x.result()
        assert not np.isnan(got).any(), f"{name} group {i}: unwritten outputs"
        assert x.guards_intact()
        assert_within_bound(got, c_ref, s_ref, f"{name} group {i}")
    # a property that holds at any size: a second launch gives the same bits
    first = [x.result().copy() for x in d]
    for x in d:
        x.reset()
    run(d)
    for f, x in zip(first, d):
        assert np.array_equal(f.view(np.uint16), x.result().view(np.uint16))


# --------------------------------------------------------- split tail tiles ---

@pytest.mark.parametrize("name", ["g2_n3072_k4096", "ragged"])
def test_small_grid_fill_matches_oracle_and_is_deterministic(name):
    # NVFP4_OPT_SPLIT_TAIL = 3 on single CTAs: fewer tiles than SMs, so the grid stays at
    # one CTA per SM and every tile is cut along K. The two-group K = 4096 set's 120 tiles
    # of 16 stages become 13 stages per CTA; the ragged set's 20 tiles of 8 stages become
    # one- or two-stage segments on every SM. Every output against the oracle, and the
    # same bits on a rerun (partials summed in K order).
    if name == "ragged":
        groups = gen.make_problem_set(44, [130, 60], [1024, 520], [2048, 2048])
    else:
        groups = gen.make_workload(name)
    nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 2)
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 3)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    assert nv.nvfp4_last_kernel() == "nvfp4_grouped_gemm_kernel<128,5>"
    check_full(groups, d, f"fill {name}")
    first = [x.result().copy() for x in d]
    for x in d:
        x.reset()
    run(d)
    for f, x in zip(first, d):
        assert np.array_equal(f.view(np.uint16), x.result().view(np.uint16))


@pytest.mark.parametrize("block_n,max_ctas", [(128, 70), (128, 72), (256, 36), (256, 37), (128, 0), (256, 7),
                                               ("pair", 38), ("pair", 40), ("pair", 0)])
def test_split_tail_tiles_match_oracle_and_are_deterministic(block_n, max_ctas):
    # Uniform K (2048 = 8 stages): 74 tiles at width 128, 38 at width 256, 21 pair tiles
    # of 256 x 256. Grids of 70/72 and 36/37 CTAs, and of 19/20 pairs, leave a short last
    # wave that is cut along K (down to one-stage segments, eight per tile, at 72 and 37
    # CTAs); the full grid and 7 CTAs do not split.
    groups = gen.make_problem_set(41, [130, 60, 200, 129], [2048, 1024, 1536, 520], [2048] * 4)
    if block_n == "pair":
        nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, 1)
        nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 2)  # pairs split only when asked to
    else:
        nv.nvfp4_set_option(nv.NVFP4_OPT_BLOCK_N, block_n)
    nv.nvfp4_set_option(nv.NVFP4_OPT_MAX_CTAS, max_ctas)
    d = [DeviceGroup(g) for g in groups]
    run(d)
    check_full(groups, d, f"split block_n={block_n} max_ctas={max_ctas}")
    first = [x.result().copy() for x in d]
    for x in d:
        x.reset()
    run(d)  # same schedule again: the same bits (partials are summed in K order)
    for f, x in zip(first, d):
        assert np.array_equal(f.view(np.uint16), x.result().view(np.uint16))
    nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 0)
    try:
        e = [DeviceGroup(g) for g in groups]
        run(e)
        check_full(groups, e, "split off")
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_SPLIT_TAIL, 1)


# ------------------------------------------------------- host threads, streams ---

def test_concurrent_calls_from_host_threads():
    # Four host threads, each with its own stream and problem set (one taking CTA pairs, one
    # single CTAs, one the swapped-operand kernel, one with row-major scales read in the
    # kernel), call the library five times each at the same time (ctypes drops the GIL).
    # The table cache, the buffer pool and the per-stream events are shared under the
    # library's lock; every output must still match the oracle.
    import threading
    specs = [(501, [200, 130, 256], [1024, 512, 768], [2048] * 3, nv.NVFP4_SF_PREPACKED),
             (502, [64, 128], [512, 384], [1024, 1024], nv.NVFP4_SF_PREPACKED),
             (503, [8, 16, 4], [1024, 512, 256], [2048, 1024, 512], nv.NVFP4_SF_PREPACKED),
             (504, [40, 129], [264, 136], [512, 1024], nv.NVFP4_SF_ROWMAJOR)]
    sets = [gen.make_problem_set(seed, Ms, Ns, Ks) for seed, Ms, Ns, Ks, _ in specs]
    devs = [[DeviceGroup(g, layout) for g in s] for s, (_, _, _, _, layout) in zip(sets, specs)]
    streams = [torch.cuda.Stream() for _ in specs]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())  # the inputs and the NaN-filled C are ready
    errors = []

    def worker(i):
        try:
            probs = [x.problem() for x in devs[i]]
            for _ in range(5):
                nv.nvfp4_grouped_gemm(probs, streams[i].cuda_stream)
        except Exception as e:  # reported below, on the test's thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(specs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert nv.nvfp4_device_status()[0] == 0
    for i, (s, d) in enumerate(zip(sets, devs)):
        check_full(s, d, f"thread {i}")
