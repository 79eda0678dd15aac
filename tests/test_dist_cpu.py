"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

With N GPUs the benchmark runs one replica of the workload per rank (the
units are independent, so there is no data-path collective); the job's time
is the slowest rank's, its throughput the work of all ranks over that time,
and only rank 0 prints.  These tests run that logic over a gloo process group
on the host, with made-up per-rank times."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world_size, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world_size), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world_size)
    try:
        assert bench.dist_env() == (world_size, rank, rank)
        # every rank gets the slowest rank's time
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        assert slowest == 10.0 + 5.0 * (world_size - 1)
        # whole-job throughput: all ranks' work over that time
        value = bench.job_throughput(2.0e12, world_size, slowest)
        assert abs(value - 2.0e12 * world_size / (slowest * 1e-3) / 1e12) < 1e-9
        # the reference arm: ranks other than 0 leave without work or output
        if rank != 0:
            assert bench.run_reference(None, None) == 0
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world_size", [2])
def test_bench_rank_logic_over_gloo(world_size):
    mp.spawn(_rank_main, args=(world_size, _free_port()), nprocs=world_size, join=True)


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for name in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(name, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_throughput(1.0e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference: the oracle on a bounded sample, one JSON line
    with the keys the benchmark contract asks for (CPU only)."""
    import json
    import subprocess
    env = dict(os.environ)
    for name in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(name, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--ref-prefix", "128", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=600, check=True)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "b2_hq32_hkv8_s8192_d128_causal_gqa"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
