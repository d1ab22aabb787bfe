"""The N > 1 host logic of bench.py, on CPU with the gloo backend (world size 2).

The hot path shards by sequence with no exchange step: every rank runs an independent
replica of the workload (its own seed) and the only cross-rank operations are the timing
barrier and the max-over-ranks of the step time. These tests run that logic in two CPU
processes: the max reduction, the whole-job rate, that the ranks' workloads differ, and
that under a two-rank launch the reference arm prints exactly one line (rank 0).
"""
import hashlib
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from sparse_attention_indexer_mqa_gb300 import workloads as W
    ms = bench.rank_max(1.0 + 0.5 * rank, world, "cpu")
    wl = W.make("tiny_decode", seed=0 + rank)
    digest = hashlib.sha256(wl.k.tobytes() + wl.q.tobytes()).hexdigest()
    digests = [None] * world
    dist.all_gather_object(digests, digest)
    with open(os.path.join(out, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "digests": digests, "pairs": wl.pairs()}, f)
    dist.destroy_process_group()


def test_rank_max_and_independent_replicas(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(r["ms"] == 1.5 for r in res)            # the slowest rank's time, on every rank
    assert res[0]["digests"] == res[1]["digests"]
    assert len(set(res[0]["digests"])) == world        # each rank has its own replica
    sys.path.insert(0, ROOT)
    import bench
    pairs = res[0]["pairs"]
    assert bench.job_rate(pairs, 1.5, world) == pytest.approx(world * pairs / 1.5e-3 / 1e3)
    assert bench.rank_max(3.0, 1, "cpu") == 3.0


def test_reference_arm_two_ranks_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--config", "tiny_decode", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_json_contract():
    """The reference arm's line carries every key of the benchmark contract (one rank, CPU)."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--config", "tiny_decode", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"] and d["config"]["pairs"] > 0
    assert {"value", "unit", "cores", "kind", "sample"} <= set(d["cpu_baseline"])
