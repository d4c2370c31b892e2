"""bench.py's host-side contract, without a GPU: the reference arm (the oracle on the host cores)
prints one JSON line for the configuration it was given, `--gpus N` starts N replica processes
(rank 0 alone reports), and a process count that disagrees with --gpus is refused."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None, timeout=600):
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          cwd=ROOT, env=env, timeout=timeout)


def _lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_reports_whole_steps_of_the_same_workload():
    r = _run(["--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    (line,) = _lines(r.stdout)
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 3
    assert line["config"]["workload"] == "tiny" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_flag_starts_that_many_replicas_and_rank0_alone_reports():
    r = _run(["--impl", "reference", "--gpus", "2", "--config", "tiny", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def test_gpus_flag_disagreeing_with_the_launch_is_refused():
    r = _run(["--impl", "reference", "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "1"],
             env_extra={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0 and "--gpus 2" in (r.stderr + r.stdout)


def test_oracle_sample_on_several_processes_covers_every_sequence():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.oracle_throughput("tiny", 2, steps=2, warmup=0)
    # two whole steps of the 4 tiny sequences, split over two processes
    assert r["seq_steps"] == 8 and r["bytes"] > 0 and r["workers"] == 2
