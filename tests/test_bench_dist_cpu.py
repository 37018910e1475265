"""The N>1 bench path on CPU: two gloo ranks reduce their timed region to
the slowest rank's, and the whole-job value counts every rank's bytes."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = 100.0 + 50.0 * rank                    # rank 1 is the slow one
    ms = bench.reduce_max_ms(my_ms, dist, device="cpu")
    val = bench.job_value(1_000_000, 10, world, ms)
    q.put((rank, ms, val))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_value():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, val in out:
        assert ms == pytest.approx(150.0)
        # 2 ranks x 10 steps x 1 MB over 0.15 s
        assert val == pytest.approx(2 * 10 * 1e6 / 0.15 / 1e9)


def test_single_rank_identity():
    import bench

    assert bench.reduce_max_ms(12.5, None) == 12.5
    assert bench.job_value(6_963_200, 100, 1, 1.0) == pytest.approx(6_963_200 * 100 / 1e-3 / 1e9)


def test_traffic_key_ignores_comments_only():
    """The recorded DRAM traffic is keyed on the kernel sources without
    comments: a comment edit keeps the key, a code edit changes it."""
    import bench

    src = "int f(int x) {  // doubles x\n  /* block\n comment */ return 2 * x;\n}\n"
    same = "// header\nint f(int x) {  // twice x\n\n  return 2 * x;\n}\n"
    other = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)


def test_committed_traffic_matches_current_sources():
    """Every recorded tensor-core entry the headline can use is keyed on the
    current sources (so the bench reports traffic, not null)."""
    import json
    import os

    import bench

    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    key = f"{bench.Q2_PATH[bench.HEADLINE['tc'][8]]}_M8_N{bench.HEADLINE['N']}_K{bench.HEADLINE['K']}"
    assert key in d
    assert bench.committed_traffic(key, bench.HEADLINE["tc"][8]) == d[key]["dram_bytes_per_launch"]
