"""The benchmark's N > 1 host logic (replicas, max-over-ranks timing,
whole-job aggregation) with world_size 2 over gloo on CPU."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    bench.dist_barrier()
    # rank r "took" 1 + r seconds to move 10 GB
    t = bench.dist_max(1.0 + r)
    q.put((r, w, t, bench.aggregate(10e9, t, w)))
    dist.destroy_process_group()


def test_dist_max_and_aggregate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, t, v in res:
        assert w == 2 and t == 2.0            # the slowest rank sets the time
        assert v == pytest.approx(10.0)       # 2 ranks x 10 GB / 2 s


def test_single_process_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.5) == 3.5
    assert bench.aggregate(4e9, 2.0, 1) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-elems", "4096"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    # the reference arm describes the very workload the GPU arm times
    sys.path.insert(0, ROOT)
    import bench
    from quantized_allreduce_codec_gb300.inputs import workloads
    assert line["config"] == bench.headline_config(workloads()[bench.HEADLINE], 1)
    assert line["config"]["W"] == 8 and line["config"]["per_rank_elems"] == 8192 * 8192
    assert line["config"]["calls_per_step"] == len(bench.STEP_CALLS) == 14


def test_bytes_alg_table():
    sys.path.insert(0, ROOT)
    import bench
    n = 1 << 20
    assert bench.bytes_alg(2, n, 0, 1, False) == 3 * 2 * n
    assert bench.bytes_alg(2, n, 3, 2, True) == 6 * n + n // 32 * 18   # Q4: 16 code bytes + scale
    assert bench.bytes_alg(8, n, 5, 2, True) == 18 * n + n // 32 * 36  # Q8 asym


def test_sampled_blocks_are_whole_distinct_and_sorted():
    sys.path.insert(0, ROOT)
    import bench
    idx = bench.sample_block_elems(1 << 16, 100, 3)
    assert idx.size == 100 * 32
    blocks = idx.reshape(-1, 32)
    assert (blocks[:, 0] % 32 == 0).all() and (blocks == blocks[:, :1] + np.arange(32)).all()
    assert (np.diff(blocks[:, 0]) > 0).all() and blocks.max() < (1 << 16)
