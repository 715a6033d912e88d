"""The bench's roofline arithmetic, checked against independent counts.

Decode bytes per token are rebuilt from the parameter count, which test_oracle_pins
checks against the page's printed figure. Each token reads every parameter once (the
LM head is the tied embedding), the token's embedding row, each layer's K and V rows of
every position, and writes fp32 logits. The FLOP counts are the rounded figures of the
long-context and short prefill workloads."""
import pytest

import bench
from synth import SHAPES, param_count


@pytest.mark.parametrize("shape,ctx", [("1p5b", 178), ("0p5b", 48), ("1p5b", 4224)])
def test_decode_bytes_per_token(shape, ctx):
    s = SHAPES[shape]
    kv_per_pos = s.n_layers * 2 * s.n_kv_heads * s.head_dim * 2  # fp16 K and V rows
    want = param_count(s) * 2 + s.hidden * 2 + kv_per_pos * ctx + s.vocab * 4
    assert bench.decode_bytes_per_token(s, ctx) == want


def test_decode_bytes_match_the_quoted_figures():
    # 1.5B at a 178-position mean context: 3093.1 MB; 0.5B at 48 positions: 989.3 MB
    assert bench.decode_bytes_per_token(SHAPES["1p5b"], 178) / 1e6 == pytest.approx(3093.1, abs=0.1)
    assert bench.decode_bytes_per_token(SHAPES["0p5b"], 48) / 1e6 == pytest.approx(989.3, abs=0.1)
    assert SHAPES["1p5b"].n_layers * 2 * SHAPES["1p5b"].n_kv_heads * SHAPES["1p5b"].head_dim * 2 == 28672


def test_gate_up_bytes_per_launch():
    s = SHAPES["1p5b"]
    assert bench.gateup_bytes(s) == 2 * 8960 * 1536 * 2 + 1536 * 2 == 55053312


@pytest.mark.parametrize("shape,P,flop", [("1p5b", 4096, 1.218e13), ("1p5b", 128, 3.37e11), ("0p5b", 32, 2.32e10)])
def test_prefill_flops(shape, P, flop):
    assert bench.prefill_flops(SHAPES[shape], P) == pytest.approx(flop, rel=2e-3)


def test_decode_launches_per_token():
    # embedding, five kernels per layer (q/k/v, attention, o_proj, gate/up, down), LM head
    assert bench.decode_launches_per_token(SHAPES["1p5b"]) == 1 + 5 * 28 + 1


def test_prefill_launch_count_matches_the_recorded_launch_lists():
    # The ncu launch lists of a 128-token and of a 4096-token prefill of the 1.5B shape
    # show, per layer: two RMSNorms, the fused q/k/v GEMM, attention, o_proj, gate/up and
    # down; at 128 tokens q/k/v, o_proj and down each add a split-K reduce (gate/up does
    # not). One embedding launch before the layers, one LM-head launch after them.
    s = SHAPES["1p5b"]
    assert bench.prefill_launches(s, 128) == 1 + s.n_layers * 10 + 1
    assert bench.prefill_launches(s, 4096) == 1 + s.n_layers * 7 + 1


def test_reference_arm_line_keeps_the_contract():
    # `bench.py --impl reference` runs the CPU oracle (float32 mode) on the 1.5B workload and
    # prints one JSON line with the contract's keys; no GPU is involved.
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([ln for ln in out.stdout.splitlines() if ln.startswith("{")][-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["dtype"] == "f32"
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == os.cpu_count() and cb["ttft_ms"] > 0 and cb["cpu"]
