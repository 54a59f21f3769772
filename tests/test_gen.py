"""The seeded input generator: determinism, distributions and the workload table."""
import os

import numpy as np

import gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_splitmix64_published_values():
    # The first outputs of splitmix64 seeded with 0 (x += GAMMA, then the finaliser),
    # as printed by Vigna's reference splitmix64.c.
    out = gen.draws(np.uint64(0), 0, 3)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_sliceable():
    a = gen.make_group(1111, 3, 40, 64, 256)
    b = gen.make_group(1111, 3, 40, 64, 256)
    for x, y in [(a.A, b.A), (a.B, b.B), (a.SFA, b.SFA), (a.SFB, b.SFB)]:
        assert np.array_equal(x, y)
    key = gen.stream_key(1111, 3, gen.TENSOR_B)
    full = gen.draws(key, 0, 5000)
    assert np.array_equal(gen.draws(key, 1234, 100), full[1234:1334])
    c = gen.make_group(1112, 3, 40, 64, 256)
    assert not np.array_equal(a.B, c.B)
    d = gen.make_group(1111, 4, 40, 64, 256)
    assert not np.array_equal(a.B, d.B)


def test_shapes_and_distributions():
    g = gen.make_group(7, 0, 256, 512, 1024)
    assert g.A.shape == (256, 512) and g.B.shape == (512, 512)
    assert g.SFA.shape == (256, 64) and g.SFB.shape == (512, 64)
    nib = np.concatenate([g.B.ravel() & 15, g.B.ravel() >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    sc = np.concatenate([g.SFA.ravel(), g.SFB.ravel()])
    assert sc.min() == 0x20 and sc.max() == 0x40
    counts = np.bincount(sc - 0x20, minlength=33)
    assert counts.min() > 0.85 * sc.size / 33 and counts.max() < 1.15 * sc.size / 33


def test_workloads_match_page_shapes():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "leaderboard_shapes.txt")) if l.strip() and not l.startswith("#")]
    page = set()
    for r in rows:
        seed = int(r[0])
        trip = tuple(tuple(int(v) for v in t.split(",")) for t in r[1:])
        page.add((seed, trip))
    ours = set()
    for name, w in gen.WORKLOADS.items():
        if name == "tiny_g2":
            continue
        ours.add((w["seed"], tuple(zip(w["Ms"], w["Ns"], w["Ks"]))))
    assert ours == page
