"""bench.py on CPU: two gloo ranks agree on the max time and pass the barrier; the reference arm
(the oracle timed on the host cores) prints one line of the contract; warm-up below 3 is refused.
(On GPUs the same functions run over NCCL. There, every rank runs its own replica and there
is no collective on the data path.)"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    bench.barrier(world)
    out[rank] = bench.reduce_max(10.0 + rank * 5.5, world)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 15.5, 1: 15.5}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_prints_one_contract_line():
    # the reference arm times the oracle on the host cores: no GPU needed
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny_g2",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us" and d["higher_is_better"] is False
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3 and d["config"]["workload"] == "tiny_g2"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_warmup_below_three_is_refused():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--warmup", "1"],
                       capture_output=True, text=True, timeout=120, cwd=root)
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr
