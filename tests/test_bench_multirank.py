"""The multi-rank path of bench.py on the CPU (gloo ranks): the slowest rank's time
sets the whole-job value, every rank sees the same maximum, only rank 0 of the
reference arm prints, and the (batch, kv head) group partition covers every group
exactly once with slices that reassemble to the whole problem (no collective on
the data path)."""
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


# ------------------------------------------------------------------ group partition
def test_group_ranges_cover_every_group_once():
    sys.path.insert(0, ROOT)
    import bench

    for total in range(0, 21):
        for world in range(1, 10):
            ranges = [bench.group_range(total, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == total
            for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
                assert a1 == b0  # contiguous, in rank order, no overlap
            sizes = [g1 - g0 for g0, g1 in ranges]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0


def _partition_rank(rank, world, port, out_dir):
    """One gloo rank of a strong partition: it computes its groups of a small problem
    with the oracle (standing in for the GPU kernel) and rank 0 reassembles them."""
    import numpy as np
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    import oracle
    from gqa_attention_forward_gb300 import workloads

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.Workload("part", 3, 4, 2, 40, 16, "bf16", True, seed=77)  # 6 groups
        sub, x, job_flops = bench.rank_problem(w, "strong", world, rank)
        o, lse, _ = oracle.attention(oracle.widen(x["q"], w.dtype), oracle.widen(x["k"], w.dtype),
                                     oracle.widen(x["v"], w.dtype), w.scale, w.causal)
        pieces = [None] * world
        dist.all_gather_object(pieces, (rank, sub.B, sub.flops, o, lse))
        if rank == 0:
            full = workloads.make_inputs(w)
            ro, rl, _ = oracle.attention(oracle.widen(full["q"], w.dtype), oracle.widen(full["k"], w.dtype),
                                         oracle.widen(full["v"], w.dtype), w.scale, w.causal)
            G = w.Hq // w.Hkv
            o_cat = np.concatenate([p[3] for p in sorted(pieces, key=lambda p: p[0])], axis=0)
            l_cat = np.concatenate([p[4] for p in sorted(pieces, key=lambda p: p[0])], axis=0)
            res = {"groups": [p[1] for p in sorted(pieces, key=lambda p: p[0])],
                   "flops_sum": sum(p[2] for p in pieces), "job_flops": job_flops,
                   "o_equal": bool(np.array_equal(o_cat.reshape(ro.shape), ro)),
                   "lse_equal": bool(np.array_equal(l_cat.reshape(rl.shape), rl)),
                   "shape": list(o_cat.shape), "G": G}
            with open(os.path.join(out_dir, "part.json"), "w") as f:
                json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_strong_partition_slices_reassemble_to_the_whole_problem(tmp_path):
    """Two gloo ranks split the 6 (batch, kv head) groups of one problem 3 + 3; their
    outputs, laid side by side in rank order, are the whole problem's outputs bit for
    bit, and their counted FLOPs add up to the problem's."""
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_partition_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r = json.load(open(tmp_path / "part.json"))
    assert r["groups"] == [3, 3]
    assert r["o_equal"] and r["lse_equal"]
    assert r["flops_sum"] == pytest.approx(r["job_flops"])
    assert r["shape"][1] == r["G"]  # each slice is laid out with Hq = G, Hkv = 1


def test_weak_partition_gives_each_rank_its_own_batch_entries():
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    from gqa_attention_forward_gb300 import workloads

    w = workloads.Workload("wk", 1, 4, 2, 32, 16, "f16", True, seed=5)
    subs = [bench.rank_problem(w, "weak", 3, r) for r in range(3)]
    for r, (sub, x, job) in enumerate(subs):
        assert sub == w and job == pytest.approx(3 * w.flops)
        ref = workloads.make_inputs(w, seed=w.seed + r)
        assert all(np.array_equal(x[n], ref[n]) for n in "qkv")
    assert not np.array_equal(subs[0][1]["q"], subs[1][1]["q"])
