"""Benchmark: batch-1 bf16 KV-cached greedy decode of the Qwen2.5-1.5B shape.

One step = one generation of the workload: prefill of a 128-token uniform-random prompt
into a 2048-position KV cache, then 99 greedy decode steps (100 tokens in total), inputs
already on the device. ``value`` is decode tokens per second over the decode portion of
the K timed steps; ``ttft_ms`` is the device time of the prefill (first token on device).
Weights are random N(0, 0.02) bf16 of the real architecture (3.09 GB, far larger than L2,
read once per token), so no L2 flush is needed between steps.

The same line carries two more sections of the same shape, each timed with its own clock
samples: ``long`` (a 4096-token prompt into an 8192-position cache: TTFT and prefill
TFLOP/s against the tensor peak, then 255 decode steps at 4096+ positions) and
``batched`` (16 sequences with prompts of 256-2048 tokens decoded together for 127 steps).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

``--impl reference`` times the CPU oracle (its float32 numpy mode) on a bounded sample of the same
workload, on the host cores. Under torchrun every rank runs its own replica of the batch-1
workloads (batch-1 decode does not shard; no collective is used on the data path), the
16 batched sequences are split over the ranks (each with a full weight replica; token ids
are gathered on the host), and rank 0 prints the line.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import SHAPES, WORKLOADS, make_prompt, make_weights  # noqa: E402

METRIC = "decode tok/s (Qwen2.5-1.5B shape, bs1, bf16)"
WORKLOAD = "1p5b"


def decode_bytes_per_token(s, ctx):
    """Algorithmic HBM bytes of one decode token: every weight once (tied LM head read
    once), the KV cache of ctx positions, the embedding row, and the fp32 logits."""
    H, I, V, L = s.hidden, s.intermediate, s.vocab, s.n_layers
    qd, kvd = s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
    e = 2 if s.dtype == "bf16" else 4
    per_layer = (H * (qd + 2 * kvd) + (qd + 2 * kvd) + qd * H + 3 * H * I + 2 * H) * e
    kv = L * 2 * kvd * ctx * e
    return L * per_layer + V * H * e + H * e + H * e + kv + V * 4


def gateup_bytes(s):
    e = 2 if s.dtype == "bf16" else 4
    return 2 * s.intermediate * s.hidden * e + s.hidden * e


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "qwen2_decoder_forward_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, src_hash):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this
    exact kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(seconds, ws, device):
    """Per entry, the largest of every rank's timings: the job is as slow as its slowest
    replica. One all-reduce of float64 values over the initialised process group."""
    if ws == 1:
        return [float(x) for x in seconds]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(units_per_rank, ws, max_seconds):
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_per_rank * ws / max_seconds


def host_cpu():
    """The host CPU's model, from /proc/cpuinfo (x86: model name; Arm: implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    for line in info:
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    fields = {}
    for line in info:
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            fields.setdefault(k, v)
    if "CPU implementer" in fields:
        return f"arm implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return "unknown"


def oracle_sample(s, wl, n_decode, warmup=0, dtype=np.float32):
    """Time the CPU oracle in its float32 mode (numpy BLAS on every host core; the precision
    of the pages' own numpy model): the workload's prompt prefill (TTFT), then decode steps.
    Returns (prefill seconds, seconds per decode step list, threads)."""
    import oracle
    w = make_weights(s)
    prompt = make_prompt(s, wl.prompt_len)
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w, dtype=dtype)
    del w
    cache = oracle.KVCache(s.n_layers)
    t0 = time.perf_counter()
    t, _ = oracle.step(om, list(prompt), np.arange(len(prompt)), cache)
    ttft = time.perf_counter() - t0
    seq = list(prompt) + [t]
    times = []
    for i in range(warmup + n_decode):
        t0 = time.perf_counter()
        t, _ = oracle.step(om, [seq[-1]], np.array([len(seq) - 1]), cache)
        dt = time.perf_counter() - t0
        seq.append(t)
        if i >= warmup:
            times.append(dt)
    return ttft, times, os.cpu_count()


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = WORKLOADS[WORKLOAD]
    s = SHAPES[wl.shape]
    ttft, times, cores = oracle_sample(s, wl, args.steps, warmup=args.warmup)
    total = sum(times)
    value = len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "Qwen2.5-1.5B shape, bs1, 128-token prompt, KV cache 2048, "
                               "greedy decode; one step = one oracle decode step after the prefill (timed apart: "
                               "cpu_baseline.ttft_ms)",
                   "global_batch": 1, "seq_len": wl.prompt_len},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle", "cpu": host_cpu(),
                         "ttft_ms": 1000 * ttft,
                         "sample": f"{len(times)} decode steps at context {wl.prompt_len}+ after the "
                                   f"{wl.prompt_len}-token prefill (timed as ttft_ms), float32 numpy (BLAS)"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def prefill_launches(s, T, nsm=152):
    """Kernels one prefill of T tokens launches on a bf16 model (the tensor-core path): the
    embedding; per layer two RMSNorms, the fused q/k/v GEMM (bias, RoPE and the KV append in
    its epilogue), attention, o_proj, gate/up (SwiGLU in its epilogue) and down, each GEMM
    followed by a split-K reduce where the planner splits K; then the LM head. Mirrors the
    GEMM planner: 64-column tiles (128 for gate/up) up to two row tiles, else 256 or 192;
    K split when the tiles leave more than half the SMs idle (gate/up: fewer than half the
    SMs' worth of tiles), at least two K blocks per split."""
    H, I = s.hidden, s.intermediate
    qd, Wd = s.n_heads * s.head_dim, (s.n_heads + 2 * s.n_kv_heads) * s.head_dim
    mt = (T + 127) // 128

    def cdiv(a, b):
        return -(-a // b)

    def splits(tiles, k):
        n = min(16, nsm // tiles, cdiv(k, 64) // 2)
        return n >= 2

    def gemm(n, k):
        if mt <= 2:
            bn = 64
        else:
            def rounds(w):
                return cdiv(mt * cdiv(n, w), nsm)
            bn = 192 if rounds(192) * 192 < rounds(256) * 256 else 256
        tiles = cdiv(n, bn) * mt
        return 1 + (1 if 2 * tiles < nsm and splits(tiles, k) else 0)

    def glu(n, k):
        tiles = cdiv(n, 64 if mt <= 2 else 128) * mt
        return 1 + (1 if tiles < nsm // 2 and splits(tiles, k) else 0)

    per_layer = 2 + 1 + gemm(Wd, H) + gemm(H, qd) + glu(I, H) + gemm(H, I)
    return 1 + s.n_layers * per_layer + 1


def decode_launches_per_token(s, persistent=False):
    """Kernels one decode step launches: the persistent decode-step kernel, or embedding,
    5 per layer and the LM head."""
    return 1 if persistent else 5 * s.n_layers + 2


def timeline_persistent(m, s, ids_dev, prompt, rank):
    """Device timeline of the persistent decode-step kernel: per phase kind, the time from
    the phase's start to its units consumed, to its end, and the grid barrier after it."""
    m.set_timeline(True)
    m.prefill_device(ids_dev.data_ptr(), len(prompt))
    kinds = ["qkv", "attn", "o_proj", "gate_up", "down"] * s.n_layers + ["lm_head"]
    n = len(kinds)
    fields = ("staged_us", "first_unit_us", "units_us", "epi_start_us", "run_us", "skew_us", "barrier_us")
    st = {k: {f: [] for f in fields} for k in set(kinds)}
    tot = []
    spread = {k: [] for k in ("qkv", "attn", "o_proj", "gate_up", "down")}
    late = {k: {} for k in spread}
    waits = {}
    import torch
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    for i in range(12):
        m.decode_steps(1)
        full = m.read_timeline().astype(np.int64)
        tl, t2, t3 = full[:n], full[n:2 * n], full[2 * n:3 * n]
        flat = full.reshape(-1)
        if i < 2:
            continue
        tot.append((tl[-1, 2] - tl[0, 0]) / 1000.0)
        for j, k in enumerate(kinds):
            if k != "attn":
                st[k]["staged_us"].append((t2[j, 0] - tl[j, 0]) / 1000.0)
                st[k]["first_unit_us"].append((t3[j, 0] - tl[j, 0]) / 1000.0)
                st[k]["units_us"].append((tl[j, 1] - tl[j, 0]) / 1000.0)
                st[k]["epi_start_us"].append((t3[j, 1] - tl[j, 0]) / 1000.0)
            st[k]["run_us"].append((tl[j, 2] - tl[j, 0]) / 1000.0)
            if j + 1 < n:
                # CTA 0's phase end -> the last CTA's arrival -> CTA 0 past the barrier
                st[k]["skew_us"].append((t2[j, 2] - tl[j, 2]) / 1000.0)
                st[k]["barrier_us"].append((t2[j, 1] - t2[j, 2]) / 1000.0)
        if len(flat) >= 9 * n + 5 * nsm + 8 * n:  # SM clock stamps of CTA 0 per phase
            cks = flat[9 * n + 5 * nsm: 9 * n + 5 * nsm + 8 * n].reshape(n, 8)
            for j, k in enumerate(kinds):
                c = cks[j]
                def d(a, b_):
                    return float(c[b_] - c[a]) if c[a] and c[b_] and c[b_] >= c[a] else float("nan")
                waits.setdefault(k, []).append((d(0, 1), d(1, 2), d(2, 3), d(3, 4), d(4, 5), d(5, 6), d(6, 7)))
        if len(flat) >= 9 * n + 5 * nsm:  # every CTA's arrival after layer 1's phases
            for kk, k in enumerate(("qkv", "attn", "o_proj", "gate_up", "down")):
                arr = flat[9 * n + kk * nsm: 9 * n + (kk + 1) * nsm]
                spread[k].append((arr.max() - arr.min()) / 1000.0)
                for b in np.argsort(arr)[-4:]:
                    late[k][int(b)] = late[k].get(int(b), 0) + 1
    m.set_timeline(False)
    out = {"persistent_step_us": float(np.mean(tot)), "phases": {
        k: {f: round(float(np.mean(x)), 3) if x else None for f, x in v.items()} for k, v in st.items()},
        "layer1_arrival_spread_us": {k: round(float(np.mean(v)), 3) if v else None for k, v in spread.items()},
        "layer1_latest_ctas": {k: sorted(v.items(), key=lambda kv: -kv[1])[:6] for k, v in late.items()},
        "cta0_cycles": {k: dict(zip(("loads", "reduce", "to_staged", "first_unit", "rest_units", "end_barrier",
                                     "epilogue"),
                                    [round(float(x), 1) for x in np.nanmean(np.array(v, dtype=float), axis=0)]))
                        for k, v in waits.items()}}
    if rank == 0:
        print(json.dumps(out), flush=True)


def timeline_per_kernel(m, s, ids_dev, prompt, rank):
    """Device timeline of single decode steps run as one kernel per operation: per kernel
    kind, the gap from the previous kernel's end to this kernel's dependency release, the
    run from release to end, and how early its CTAs were resident."""
    m.set_timeline(True)
    m.prefill_device(ids_dev.data_ptr(), len(prompt))
    kinds = ["embed"] + ["qkv", "attn", "o_proj", "gate_up", "down"] * s.n_layers + ["lm_head"]
    stats = {k: {"gap_us": [], "run_us": [], "early_us": []} for k in set(kinds)}
    totals = []
    for i in range(12):
        m.decode_steps(1)
        tl = m.read_timeline().astype(np.int64)
        if i < 2:
            continue
        totals.append((tl[-1, 2] - tl[0, 0]) / 1000.0)
        for j, k in enumerate(kinds):
            prev_end = tl[j - 1, 2] if j else tl[0, 0]
            stats[k]["gap_us"].append((tl[j, 1] - prev_end) / 1000.0)
            stats[k]["run_us"].append((tl[j, 2] - tl[j, 1]) / 1000.0)
            stats[k]["early_us"].append((tl[j, 1] - tl[j, 0]) / 1000.0)
    m.set_timeline(False)
    out = {"timeline_step_us": float(np.mean(totals)), "kernels": {}}
    for k, v in stats.items():
        out["kernels"][k] = {f: round(float(np.mean(x)), 3) for f, x in v.items()}
        out["kernels"][k]["per_step_us"] = round(float(np.sum(v["run_us"]) + np.sum(v["gap_us"])) / len(totals), 2)
    if rank == 0:
        print(json.dumps(out), flush=True)



def run_native(args):
    import torch
    import __graft_entry__
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    __graft_entry__.build()
    from qwen2_decoder_forward_decode_gb300 import DeviceWeights, Model

    torch.cuda.set_device(local)
    wl = WORKLOADS[WORKLOAD]
    s = SHAPES[wl.shape]
    if args.layers:
        import dataclasses
        s = dataclasses.replace(s, n_layers=args.layers)
    n_dec = wl.new_tokens - 1
    w = make_weights(s)
    dw = DeviceWeights(w, 1)
    prompt = make_prompt(s, wl.prompt_len)
    stream = torch.cuda.Stream()
    m = Model(s, dw, wl.kv_capacity, stream=stream.cuda_stream)
    ids_dev = torch.from_numpy(prompt).to(f"cuda:{local}")
    torch.cuda.synchronize()

    def one_step():
        m.prefill_device(ids_dev.data_ptr(), len(prompt))
        m.decode_steps(n_dec)

    for _ in range(args.warmup):
        one_step()
    m.sync()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_host0 = time.perf_counter()
        for k in range(args.steps):
            ev[k][0].record(stream)
            m.prefill_device(ids_dev.data_ptr(), len(prompt))
            ev[k][1].record(stream)
            m.decode_steps(n_dec)
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        t_host = time.perf_counter() - t_host0
    if ws > 1:
        torch.distributed.barrier()
    m.sync()
    prefill_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps)]
    decode_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(args.steps)]
    step_ms = [ev[k][0].elapsed_time(ev[k][2]) for k in range(args.steps)]
    dec_s, tot_s = max_over_ranks([sum(decode_ms) / 1000.0, sum(step_ms) / 1000.0], ws, f"cuda:{local}")
    value = job_throughput(n_dec * args.steps, ws, dec_s)
    ctx_mean = wl.prompt_len + (n_dec - 1) / 2.0 + 1  # positions read per decode token, mean
    bpt = decode_bytes_per_token(s, ctx_mean)
    peak, peak_kind = read_peaks()

    # ---- dominant kernel (gate/up GEMV, 59% of a layer's bytes) timed with CUDA events
    # around every layer's launch, over a traced pass of decode steps right after the
    # timed region (the traced kernel runs without PDL overlap).
    begin = [torch.cuda.Event(enable_timing=True) for _ in range(s.n_layers)]
    end = [torch.cuda.Event(enable_timing=True) for _ in range(s.n_layers)]
    for e in begin + end:  # torch creates the CUDA event at its first record
        e.record(stream)
    stream.synchronize()
    m.set_trace(3, begin, end)
    m.prefill_device(ids_dev.data_ptr(), len(prompt))
    kt = []
    for i in range(16):
        m.decode_steps(1)
        stream.synchronize()
        if i >= 2:
            kt += [b.elapsed_time(e) for b, e in zip(begin, end)]
    m.set_trace(3, None, None)
    gu_ms = float(np.mean(kt))
    gu_bytes = gateup_bytes(s)
    src = source_hash()
    persistent = m.decode_kernels_per_step() == 1
    if persistent:
        # the dominant kernel is the decode-step kernel itself: one launch per token, timed
        # with CUDA events on its stream around the timed decode loop
        roofline = {"bound": "hbm", "kernel": "decode_step_kernel", "achieved": bpt * value / ws / 1e9,
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": bpt * value / ws / 1e9 / peak,
                    "traffic": recorded_traffic("decode_step_kernel", src), "algorithmic_bytes_per_launch": bpt,
                    "launch_us": 1e6 * ws / value,
                    "timing": "CUDA events on the decode stream around the timed decode loop (one launch per token)",
                    "gateup_gemv_us_one_kernel_per_op": gu_ms * 1000.0}
    else:
        achieved = gu_bytes / (gu_ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "kernel": "gateup_gemv", "achieved": achieved,
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": recorded_traffic("gateup_gemv", src),
                    "algorithmic_bytes_per_launch": gu_bytes, "launch_us": gu_ms * 1000.0}

    if args.timeline:
        if persistent:
            timeline_persistent(m, s, ids_dev, prompt, rank)
        else:
            timeline_per_kernel(m, s, ids_dev, prompt, rank)

    if args.layers:
        # profiling run on a reduced stack: timed loop only, not a bench line
        if rank == 0:
            print(json.dumps({"profile_run": True, "layers": s.n_layers, "decode_tok_s": value,
                              "gateup_us": gu_ms * 1000.0}), flush=True)
        m.close()
        return

    # ---- end to end through the public API with host buffers (qw_generate: H2D of the
    # prompt, prefill, decode loop, D2H of the tokens) and host-side TTFT (qw_prefill).
    e2e_steps = max(1, min(args.steps, 5))
    t_gen, t_pref = [], []
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        toks = m.generate(prompt, wl.new_tokens)
        t_gen.append(time.perf_counter() - t0)
        assert len(toks) == wl.new_tokens
        t0 = time.perf_counter()
        m.prefill(prompt)
        t_pref.append(time.perf_counter() - t0)
    e2e_decode_s = max(1e-9, float(np.mean(t_gen)) - float(np.mean(t_pref)))
    e2e_decode_s, = max_over_ranks([e2e_decode_s], ws, f"cuda:{local}")
    e2e_value = job_throughput(n_dec, ws, e2e_decode_s)

    # ---- the other two workloads of the same shape, each with its own clock samples:
    # long context (TTFT of a 4096-token prompt on the tensor cores, decode at 4096+
    # positions) and batched decode of 16 sequences
    sec_steps, sec_warm = max(1, min(args.steps, 5)), 3
    long_sec = batched_sec = None
    if not args.headline_only:
        long_sec = measure_long(dw, s, sec_steps, sec_warm, ws, local)
        batched_sec = measure_batched(dw, s, sec_steps, sec_warm, ws, rank, local)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        ttft, times, cores = oracle_sample(s, wl, 5)
        cpu = {"value": len(times) / sum(times), "unit": "tok/s", "cores": cores, "kind": "oracle",
               "cpu": host_cpu(), "ttft_ms": 1000 * ttft,
               "sample": f"the {wl.prompt_len}-token prefill (ttft_ms) and 5 decode steps, float32 numpy "
                         "(BLAS, every host core; same weights, prompt and cache length)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random N(0,0.02) bf16 weights, uniform-random prompt ids)",
            "config": {"workload": "Qwen2.5-1.5B shape (28 layers, hidden 1536, 12/2 heads, "
                                   "head_dim 128, MLP 8960, vocab 151936, tied), bs1, 128-token "
                                   "prompt, 100 greedy tokens, KV cache 2048",
                       "global_batch": ws, "seq_len": wl.prompt_len,
                       "parallelism": "replicas" if ws > 1 else "single",
                       "l2": "inputs larger than L2 (3.09 GB of weights per token)",
                       "step": "prefill + 99 decode steps; value counts decode tokens over decode time"},
            "ttft_ms": float(np.mean(prefill_ms)),
            "hbm_gbs": bpt * value / ws / 1e9,
            "decode_bytes_per_token": bpt,
            "decode_frac_of_hbm_peak": bpt * value / ws / 1e9 / peak,
            "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": 4 * wl.prompt_len,
                    "d2h_bytes_per_step": 4 * wl.new_tokens + 4,
                    "how": "qw_generate with host buffers minus qw_prefill with host buffers, host wall clock",
                    "generate_ms": 1000 * float(np.mean(t_gen)), "ttft_ms": 1000 * float(np.mean(t_pref))},
            "gpu_launches": args.steps * (prefill_launches(s, wl.prompt_len) +
                                          decode_launches_per_token(s, persistent) * n_dec),
            "clocks": clk.summary(),
            "host_ms_per_step": 1000 * t_host / args.steps,
            "source_hash": src,
        }
        if long_sec:
            line["long"] = long_sec
        if batched_sec:
            line["batched"] = batched_sec
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    m.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


def shard_sequences(n_seqs, rank, ws):
    """Sequences of the batched workload that rank `rank` of `ws` decodes: b with
    b % ws == rank. Sequences are independent (no cross-sequence attention), so ranks
    share nothing but the weights, which every rank holds in full."""
    return [b for b in range(n_seqs) if b % ws == rank]


def gather_tokens(mine, tokens, ws, n_seqs):
    """Host-side gather of every rank's token ids: `mine` are this rank's sequence indices
    and `tokens` their token lists. Returns the n_seqs lists in sequence order, on every
    rank (one all_gather_object over the process group; nothing when ws == 1)."""
    parts = [(list(mine), [list(map(int, t)) for t in tokens])]
    if ws > 1:
        import torch.distributed as dist
        parts = [None] * ws
        dist.all_gather_object(parts, (list(mine), [list(map(int, t)) for t in tokens]))
    out = [None] * n_seqs
    for idx, toks in parts:
        for b, t in zip(idx, toks):
            assert out[b] is None, f"sequence {b} decoded by two ranks"
            out[b] = t
    assert all(t is not None for t in out), "a sequence was decoded by no rank"
    return out


def measure_batched(dw, s, steps, warmup, ws, rank, local, timeline=False):
    """Batched decode of the 16-sequence workload (prompt lengths uniform in 256..2048,
    128 tokens each, KV cache 2304): prefill every sequence, then 127 decode steps of all
    of them together. Under several ranks the sequences are split over the ranks
    (shard_sequences): each rank decodes its share with a full weight replica and the
    token ids are gathered on the host. Returns the section of the bench line."""
    import torch
    from qwen2_decoder_forward_decode_gb300 import Model
    from synth import make_batch_prompts

    wl = WORKLOADS["1p5b_batch"]
    n_all, n_dec = wl.n_seqs, wl.new_tokens - 1
    prompts_all = make_batch_prompts(s, n_all, *wl.batch_len_range)
    mine = shard_sequences(n_all, rank, ws)
    prompts = [prompts_all[b] for b in mine]
    B = len(prompts)
    stream = torch.cuda.Stream()
    m = Model(s, dw, wl.kv_capacity, max_seqs=B, stream=stream.cuda_stream)
    ids = [torch.from_numpy(p).to(f"cuda:{local}") for p in prompts]
    torch.cuda.synchronize()

    def prefill_all():
        for b in range(B):
            m.prefill_device(ids[b].data_ptr(), len(prompts[b]), seq=b)

    for _ in range(warmup):
        prefill_all()
        m.decode_steps(n_dec)
    m.sync()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for k in range(steps):
            ev[k][0].record(stream)
            prefill_all()
            ev[k][1].record(stream)
            m.decode_steps(n_dec)
            ev[k][2].record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    m.sync()
    dec_s = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(steps)) / 1000.0
    pre_s = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(steps)) / 1000.0
    dec_s, pre_s = max_over_ranks([dec_s, pre_s], ws, f"cuda:{local}")
    tl_out = batched_timeline(m, s, prefill_all) if timeline else None
    # one more step outside the timed region returns every sequence's next token on the
    # host; the ranks' token ids are gathered there
    last = m.decode_step()[:B]
    gathered = gather_tokens(mine, [[t] for t in last], ws, n_all)
    m.close()
    lens = np.array([len(p) for p in prompts_all], dtype=np.float64)
    ctx_mean = lens + (n_dec - 1) / 2.0 + 1  # positions read per sequence, mean over steps
    # algorithmic bytes of one step of the whole job: every rank reads the weights once,
    # plus each sequence's KV rows, plus the logits
    weights = decode_bytes_per_token(s, 0) - s.vocab * 4
    kv = sum(decode_bytes_per_token(s, c) - decode_bytes_per_token(s, 0) for c in ctx_mean)
    step_bytes = ws * weights + kv + n_all * s.vocab * 4
    step_s = dec_s / (n_dec * steps)
    peak, peak_kind = read_peaks()
    tokens = n_all * n_dec * steps
    return {"workload": "Qwen2.5-1.5B shape, 16 sequences, prompts 256-2048 tokens (seed 2), 128 tokens "
                        "each, KV cache 2304 per sequence",
            "value": tokens / dec_s, "unit": "tok/s", "steps": steps, "warmup": warmup,
            "ms_per_decode_step": 1000.0 * step_s, "prefill_tok_s": float(lens.sum()) * steps / pre_s,
            "bytes_per_step": step_bytes, "achieved_gbs": step_bytes / step_s / 1e9 / ws,
            "peak_gbs": peak, "peak_kind": peak_kind,
            "frac_of_hbm": step_bytes / step_s / 1e9 / ws / peak,
            "sequences_per_rank": B, "parallelism": f"sequences split over {ws} ranks" if ws > 1 else "single",
            "scaling": "strong", "gathered_sequences": sum(1 for t in gathered if t), "clocks": clk.summary(),
            **({"timeline": tl_out} if tl_out else {})}


def batched_timeline(m, s, prefill_all):
    """Device timeline of single batched steps: per kernel kind, the run from dependency
    release to end and the gap from the previous kernel's end."""
    import torch
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    # SwiGLU runs in the gate/up GEMM's epilogue when its 64-row tiles cover half the SMs
    glu = os.environ.get("QW_BATCHED_GLU") != "0" and 2 * ((s.intermediate + 63) // 64) >= nsm
    layer = ["qkv_gemm", "qkv_epi", "attn", "attn_merge", "o_gemm", "o_resid_norm", "gu_gemm"]
    layer += ([] if glu else ["swiglu"]) + ["down_gemm", "down_resid_norm"]
    kinds = ["embed_norm"] + layer * s.n_layers + ["lm_gemm", "finalize"]
    m.set_timeline(True)
    prefill_all()
    st = {k: {"gap_us": [], "run_us": []} for k in set(kinds)}
    tot = []
    for i in range(8):
        m.decode_steps(1)
        tl = m.read_timeline().astype(np.int64)[:len(kinds)]
        if i < 2:
            continue
        tot.append((tl[-1, 2] - tl[0, 0]) / 1000.0)
        for j, k in enumerate(kinds):
            prev_end = tl[j - 1, 2] if j else tl[0, 0]
            st[k]["gap_us"].append((tl[j, 1] - prev_end) / 1000.0)
            st[k]["run_us"].append((tl[j, 2] - tl[j, 1]) / 1000.0)
    m.set_timeline(False)
    return {"step_us": float(np.mean(tot)), "kernels": {
        k: {"run_us": round(float(np.mean(v["run_us"])), 3), "gap_us": round(float(np.mean(v["gap_us"])), 3),
            "per_step_us": round(float(np.sum(v["run_us"]) + np.sum(v["gap_us"])) / len(tot), 1)}
        for k, v in st.items()}}


def prefill_flops(s, P):
    """Algorithmic FLOP of a P-token prefill: the linear layers on every row, causal
    attention (q.k and p.v over j <= i), and the LM head on the last row."""
    H, I, V, L = s.hidden, s.intermediate, s.vocab, s.n_layers
    qd, kvd = s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
    linear = 2 * P * L * (H * (qd + 2 * kvd) + qd * H + 3 * H * I)
    attn = 2 * 2 * s.n_heads * s.head_dim * L * P * (P + 1) / 2
    return linear + attn + 2 * V * H


def measure_long(dw, s, steps, warmup, ws, local):
    """Long-context single sequence (4096-token prompt, 256 tokens, KV cache 8192): TTFT,
    prefill throughput against the tensor peak, and decode throughput. Every rank runs its
    own replica. Returns the section of the bench line."""
    import torch
    from qwen2_decoder_forward_decode_gb300 import Model

    wl = WORKLOADS["1p5b_long"]
    n_dec = wl.new_tokens - 1
    prompt = make_prompt(s, wl.prompt_len)
    stream = torch.cuda.Stream()
    m = Model(s, dw, wl.kv_capacity, stream=stream.cuda_stream)
    ids_dev = torch.from_numpy(prompt).to(f"cuda:{local}")
    torch.cuda.synchronize()
    for _ in range(warmup):
        m.prefill_device(ids_dev.data_ptr(), len(prompt))
        m.decode_steps(n_dec)
    m.sync()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for k in range(steps):
            ev[k][0].record(stream)
            m.prefill_device(ids_dev.data_ptr(), len(prompt))
            ev[k][1].record(stream)
            m.decode_steps(n_dec)
            ev[k][2].record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    m.sync()
    m.close()
    pre_s = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(steps)) / 1000.0
    dec_s = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(steps)) / 1000.0
    pre_s, dec_s = max_over_ranks([pre_s, dec_s], ws, f"cuda:{local}")
    fl = prefill_flops(s, wl.prompt_len)
    ctx_mean = wl.prompt_len + (n_dec - 1) / 2.0 + 1
    bpt = decode_bytes_per_token(s, ctx_mean)
    peak, peak_kind = read_peaks()
    tpeak, tpeak_kind = read_tensor_peak()
    ttft = pre_s / steps
    dec_rate = job_throughput(n_dec * steps, ws, dec_s)
    return {"workload": "Qwen2.5-1.5B shape, bs1, 4096-token prompt, 256 tokens, KV cache 8192",
            "steps": steps, "warmup": warmup, "ttft_ms": 1000.0 * ttft, "prefill_flop": fl,
            "prefill_tflops": fl / ttft / 1e12, "tensor_peak_tflops": tpeak, "tensor_peak_kind": tpeak_kind,
            "prefill_frac_of_tensor_peak": fl / ttft / 1e12 / tpeak,
            "decode_tok_s": dec_rate, "decode_bytes_per_token": bpt,
            "decode_frac_of_hbm": bpt * dec_rate / ws / 1e9 / peak, "peak_gbs": peak, "peak_kind": peak_kind,
            "clocks": clk.summary()}


def read_tensor_peak():
    """Dense fp16/bf16 tensor peak (TFLOP/s) for a prefill timed in isolation: the burst
    figure of the measured peaks, else the fallback (fp16 and bf16 share the rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            v = json.load(f).get("bf16_tflops")
        if v:
            return float(v), "measured (bf16 dense burst; fp16 operands run at the same rate)"
    return 1900.0, "fallback"


def measure_gemms(s, M, reps=20):
    """Profiling: the prefill projections of one layer of shape s for an M-token prompt, each
    timed alone through the GEMM entry points (CUDA events, `reps` launches back to back)."""
    import torch
    from qwen2_decoder_forward_decode_gb300 import binding
    H, I = s.hidden, s.intermediate
    qkv = (s.n_heads + 2 * s.n_kv_heads) * s.head_dim
    shapes = [("qkv", qkv, H, True, False), ("o_proj", H, s.n_heads * s.head_dim, False, True),
              ("gate_up", I, H, None, None), ("down", H, I, False, True)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    out = {}
    for name, N, K, bias, acc in shapes:
        A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).half()
        if name == "gate_up":
            Wg = (torch.randn(N, K, device="cuda", generator=g) * 0.02).half()
            Wu = (torch.randn(N, K, device="cuda", generator=g) * 0.02).half()
            act = torch.empty(M, N, dtype=torch.float16, device="cuda")
            f = lambda: binding.gemm_swiglu_f16(M, N, K, A.data_ptr(), Wg.data_ptr(), Wu.data_ptr(),
                                                act.data_ptr(), err.data_ptr())
            flop = 2.0 * M * 2 * N * K
        else:
            B = (torch.randn(N, K, device="cuda", generator=g) * 0.02).half()
            bb = (torch.randn(N, device="cuda", generator=g) * 0.02).bfloat16()
            C = torch.zeros(M, N, device="cuda")
            f = lambda: binding.gemm_f16(M, N, K, A.data_ptr(), B.data_ptr(), bb.data_ptr() if bias else None,
                                         C.data_ptr(), acc, err.data_ptr())
            flop = 2.0 * M * N * K
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            f()
        e1.record()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, "device error bits set"
        us = e0.elapsed_time(e1) * 1000.0 / reps
        out[name] = {"N": N, "K": K, "us": us, "tflops": flop / us / 1e6}
    return out


def run_section(args):
    """Profiling: one of the extra workloads alone (one JSON line, not the bench line)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from qwen2_decoder_forward_decode_gb300 import DeviceWeights
    torch.cuda.set_device(0)
    s = SHAPES["1p5b"]
    if args.layers:
        import dataclasses
        s = dataclasses.replace(s, n_layers=args.layers)
    if args.gemm:
        peak, kind = read_tensor_peak()
        out = {"profile_run": "gemm", "M": 4096, "shape": s.name, "gemms": measure_gemms(s, 4096),
               "tensor_peak_tflops": peak, "tensor_peak_kind": kind}
        for v in out["gemms"].values():
            v["frac_of_tensor_peak"] = v["tflops"] / peak
        print(json.dumps(out), flush=True)
        return
    dw = DeviceWeights(make_weights(s), 1)
    if args.long:
        out = measure_long(dw, s, args.steps, args.warmup, 1, 0)
    else:
        out = measure_batched(dw, s, args.steps, args.warmup, 1, 0, 0, timeline=args.timeline)
    out["profile_run"] = "long" if args.long else "batched"
    out["layers"] = s.n_layers
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the long-context and batched sections of the bench line")
    ap.add_argument("--timeline", action="store_true",
                    help="also print a device timeline summary of single decode steps")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: build the 1.5B shape with this many layers")
    ap.add_argument("--batched", action="store_true",
                    help="profiling: only the batched section (one JSON line, not the bench line)")
    ap.add_argument("--long", action="store_true",
                    help="profiling: only the long-context section (one JSON line, not the bench line)")
    ap.add_argument("--gemm", action="store_true",
                    help="profiling: the prefill projections of one layer at 4096 tokens, each timed alone")
    args = ap.parse_args()
    if args.long or args.batched or args.gemm:
        run_section(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
