"""The benchmark's multi-rank path on CPU: two gloo ranks (no GPU).

Each rank is an independent replica (its own batch, no data-path exchange);
the only cross-rank steps are the barrier around the timed region and the
max over ranks of its length.  The reference arm runs on rank 0 alone.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        assert (r, w) == (rank, world)
        batch = bench.make_batch("gqa_8b", rank)
        bench.barrier(world)
        slowest = bench.max_over_ranks(1.0 + rank, world)   # rank r "took" 1 + r seconds
        value = bench.weak_scaling_value(batch.num_seqs, world, 10, slowest)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value, "seed": batch.seed,
                       "lens_sum": int(batch.context_lens.sum()),
                       "tables0": batch.block_tables[0, :4].tolist()}, f)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_are_independent_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    assert r[0]["slowest"] == r[1]["slowest"] == 2.0        # max over ranks
    assert r[0]["value"] == r[1]["value"] == 128 * 2 * 10 / 2.0
    assert r[0]["seed"] != r[1]["seed"]                      # independent batches
    assert (r[0]["lens_sum"], r[0]["tables0"]) != (r[1]["lens_sum"], r[1]["tables0"])


def test_reference_arm_under_torchrun_prints_once():
    """``torchrun --nproc-per-node 2 bench.py --impl reference``: rank 0 prints
    one JSON line, rank 1 exits 0 without work."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


@pytest.mark.parametrize("workload", ["prefix_8b", "sampling_8b", "prefill_8b", "block_copy_8b",
                                      "swap_8b", "pool_churn"])
def test_reference_arm_prints_one_complete_line(workload):
    """``bench.py --impl reference --workload W``: the oracle arm of every
    bench workload prints one JSON line with the contract's keys, the
    workload's name and a positive value (CPU only)."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           workload, "--steps", "1", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"].startswith(workload.split("_")[0])


def test_pool_churn_arms_drive_the_same_stream():
    """``bench.py --workload pool_churn`` runs on the host alone; the native
    pool and the oracle's model of it take the same steps on the same request
    stream and end with the same prefix hits and evictions (CPU only)."""
    lines = []
    for extra in ([], ["--impl", "reference"]):
        cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "pool_churn",
               "--steps", "1", "--warmup", "3"] + extra
        out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
        assert out.returncode == 0, out.stderr[-2000:]
        lines.append(json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1]))
    nat, ref = lines
    assert "impl" not in nat and ref["impl"] == "reference"
    assert nat["steps"] == ref["steps"] > 0
    for key in ("prefix_hit_tokens", "evictions"):
        assert nat["config"][key] == ref["config"][key], key
    assert nat["config"]["prefix_hit_tokens"] > 0


@pytest.mark.parametrize("workload,cascade", [("mha_7b", False), ("gqa_8b", False),
                                              ("sampling_8b", True)])
def test_reference_arm_config_and_warmup_match_the_measured_arm(workload, cascade):
    """The reference arm prints the measured arm's ``config`` (built by the
    same function from the same batch) and the requested warm-up count."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           workload, "--steps", "1", "--warmup", "4"] + (["--cascade"] if cascade else [])
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    batch = bench.make_batch(workload, 0, model_pool=True)
    want = bench.cascade_config(batch) if cascade else bench.decode_config(batch, 1)
    assert line["config"] == json.loads(json.dumps(want))
    assert line["warmup"] == 4 and line["steps"] == 1
