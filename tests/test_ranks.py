"""The bench's replica path under several ranks, on CPU (gloo, world size 2).

Batch-1 decode does not shard, so every rank runs its own replica:
- the job's time is the slowest rank's;
- its throughput counts every rank's tokens;
- the reference arm runs on rank 0 alone."""
import argparse
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:" + sys.argv[2],
                        rank=int(sys.argv[3]), world_size=2)
rank = dist.get_rank()
dist.barrier()
# rank r took 1 + r seconds to decode and 5 - r seconds per step
dec_s, tot_s = bench.max_over_ranks([1.0 + rank, 5.0 - rank], 2, "cpu")
value = bench.job_throughput(99, 2, dec_s)
dist.barrier()
print(json.dumps({"rank": rank, "dec_s": dec_s, "tot_s": tot_s, "value": value}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_slowest_rank_sets_the_job_time():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", WORKER, ROOT, str(port), str(r)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        try:
            outs.append(p.communicate(timeout=120))
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1]
    for r in res:  # every rank sees the same maxima
        assert r["dec_s"] == 2.0 and r["tot_s"] == 5.0
        assert r["value"] == pytest.approx(99 * 2 / 2.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([0.5, 1.5], 1, "cpu") == [0.5, 1.5]
    assert bench.job_throughput(99, 1, 0.5) == pytest.approx(198.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(gpus=2, steps=1, warmup=0)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
