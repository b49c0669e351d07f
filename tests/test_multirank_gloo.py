"""Host logic of the multi-GPU (replicas only) benchmark path, as world-size-2
gloo ranks on CPU: the whole-job time is the slowest rank's, and the value
counts the tokens of every replica."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    local_ms = 100.0 + 50.0 * rank          # rank 1 is slower
    res = bench.aggregate_over_ranks(local_ms, 32768, 10, world, None)
    with open(os.path.join(out_dir, "r%d.txt" % rank), "w") as f:
        f.write(" ".join(repr(v) for v in res))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks(tmp_path):
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        max_ms, ms_per_step, tps = map(float, open(tmp_path / ("r%d.txt" % rank)).read().split())
        assert max_ms == 150.0
        assert ms_per_step == 15.0
        assert tps == pytest.approx(2 * 32768 / 0.015)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
