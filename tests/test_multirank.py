"""Host logic of bench.py's N-process path, run as two gloo ranks on the CPU.

The path shards by sequence with no exchange (every rank decodes its own
batch), so the only cross-rank step is the timing reduction: whole-job
throughput = the units all ranks processed / the slowest rank's time.  Each
rank is a separate process launched with the environment torchrun sets
(RANK, WORLD_SIZE, MASTER_ADDR, MASTER_PORT)."""
import argparse
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

RANK_CODE = r"""
import json, os, sys
sys.path.insert(0, os.environ["BENCH_ROOT"])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
# rank r processed 100 (r + 1) tokens in 10 (r + 1) ms
rate, slow = bench.job_rate(10.0 * (r + 1), 100 * (r + 1))
print(json.dumps({"rank": r, "rate": rate, "slow_ms": slow}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code, ws, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(ws):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(ws),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), BENCH_ROOT=ROOT)
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            out, err = p.communicate()
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_job_rate_is_all_units_over_the_slowest_rank():
    outs = _launch(RANK_CODE, 2)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    for r in res:
        # every rank sees the same job figures: 300 tokens over 20 ms
        assert r["slow_ms"] == 20.0
        assert r["rate"] == pytest.approx(300 / 0.020)


def test_job_rate_without_a_process_group_is_the_local_rate():
    rate, ms = bench.job_rate(10.0, 100)
    assert ms == 10.0 and rate == pytest.approx(10000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the oracle arm prints one line from rank 0; the other
    ranks exit without work (checked here without starting the oracle)."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload="v2_b16_ctx4k", seed=0, steps=1, warmup=0,
                              impl="reference", gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
