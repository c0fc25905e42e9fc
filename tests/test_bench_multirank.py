"""The multi-rank path of bench.py on the CPU: two gloo ranks, each with its own
replica (weak scaling, no collective on the data path).  The slowest rank's time
sets the whole-job value, every rank sees the same maximum, and only rank 0 of
the reference arm prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [7.0, 11.5][rank]  # rank 1 is the slow one
        worst = bench.max_over_ranks(my_ms)
        value = bench.whole_job_tflops(1e12, 10, world, worst)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"worst": worst, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(2)]
    assert r[0]["worst"] == r[1]["worst"] == 11.5
    # 2 ranks x 10 steps x 1e12 FLOP over the slowest rank's 11.5 ms
    assert r[0]["value"] == pytest.approx(2 * 10 * 1e12 / 11.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_tflops(2e12, 4, 1, 8.0) == pytest.approx(1000.0)


def test_reference_arm_prints_on_rank_0_only(tmp_path):
    """bench.py --impl reference under two ranks: rank 1 exits 0 without output; rank 0
    prints one JSON line (the float64 oracle on a small row sample)."""
    outs = []
    for rank in (1, 0):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
        p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--workload", "tiny_causal_gqa_f16", "--steps", "2", "--warmup", "1"],
                           env=env, capture_output=True, text=True, timeout=300)
        assert p.returncode == 0, p.stderr
        outs.append(p.stdout.strip())
    assert outs[0] == ""
    line = json.loads(outs[1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
