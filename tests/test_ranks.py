"""The bench's multi-rank paths, on CPU (gloo, world size 2).

Batch-1 decode does not shard, so every rank runs its own replica:
- the job's time is the slowest rank's;
- its throughput counts every rank's tokens;
- the reference arm runs on rank 0 alone.
Batched decode splits its independent sequences over the ranks:
- every sequence is decoded by exactly one rank;
- the token ids gathered on the host equal a one-rank run of the same seeds."""
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


SHARD_WORKER = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch.distributed as dist
import bench, oracle
from synth import SHAPES, make_weights, make_batch_prompts
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:" + sys.argv[2],
                        rank=int(sys.argv[3]), world_size=2)
rank = dist.get_rank()
s = SHAPES["tiny"]
om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), make_weights(s))
prompts = make_batch_prompts(s, 5, 3, 9)
mine = bench.shard_sequences(5, rank, 2)
# the decoder of each rank's share: the oracle stands in for the device here
toks = [oracle.generate(om, prompts[b], 4)[0] for b in mine]
out = bench.gather_tokens(mine, toks, 2, 5)
print(json.dumps({"rank": rank, "mine": mine, "tokens": out}))
dist.destroy_process_group()
"""


def test_sequence_sharding_covers_every_sequence_once_and_gathers_the_one_rank_result():
    import oracle
    from synth import SHAPES, make_batch_prompts, make_weights
    import bench
    parts = [bench.shard_sequences(16, r, 3) for r in range(3)]
    assert sorted(b for p in parts for b in p) == list(range(16))
    assert bench.shard_sequences(16, 0, 1) == list(range(16))
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", SHARD_WORKER, ROOT, str(port), str(r)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        try:
            outs.append(p.communicate(timeout=180))
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda r: r["rank"])
    assert res[0]["mine"] == [0, 2, 4] and res[1]["mine"] == [1, 3]
    s = SHAPES["tiny"]
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), make_weights(s))
    prompts = make_batch_prompts(s, 5, 3, 9)
    one_rank = bench.gather_tokens(list(range(5)), [oracle.generate(om, p, 4)[0] for p in prompts], 1, 5)
    for r in res:  # every rank holds the full, ordered result
        assert r["tokens"] == one_rank


def test_gather_rejects_a_sequence_decoded_twice_or_never():
    import bench
    with pytest.raises(AssertionError):
        bench.gather_tokens([0, 0], [[1], [2]], 1, 2)
    with pytest.raises(AssertionError):
        bench.gather_tokens([0], [[1]], 1, 2)
