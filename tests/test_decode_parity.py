"""Parity of the CUDA path (through the C ABI) with the CPU oracle, under teacher forcing.

Small shapes run the full generation; the Qwen2.5-0.5B workload runs in full; the
Qwen2.5-1.5B workloads (128-token prompt / 2048 cache, 4096-token prompt / 8192 cache)
compare the prefill and a sample of decode steps, in the launch configuration the bench
uses (CUDA-graph decode steps with programmatic dependent launch).
"""
import numpy as np
import pytest

import oracle
from parity import check_step, oracle_run, record, run_teacher_forced, StepReport
from synth import SHAPES, WORKLOADS, make_prompt, make_weights

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _model(shape_name, w, cap, max_seqs=1):
    from qwen2_decoder_forward_decode_gb300 import DeviceWeights, Model
    s = SHAPES[shape_name]
    dw = DeviceWeights(w, 1 if s.dtype == "bf16" else 0)
    return Model(s, dw, cap, max_seqs=max_seqs)


@pytest.mark.parametrize("shape_name,P,n_new,cap", [
    ("tiny", 8, 8, 16),          # the tiny workload: 8-token prompt, 8 tokens, cache 16
    ("small_f32", 37, 20, 64),   # ragged K (96, 200), 3 query heads per KV head, head_dim 32
    ("mha_f32", 70, 10, 96),     # n_kv_heads == n_heads, prompt spans two attention tiles
    ("small_bf16", 100, 40, 160),
    ("hd128_bf16", 150, 12, 200),
    ("untied_bf16", 45, 12, 64),  # separate LM head, no q/k/v bias, vocab 2051
])
def test_small_shapes_teacher_forced(shape_name, P, n_new, cap):
    w, prompt, toks, logits = oracle_run(shape_name, P, n_new)
    m = _model(shape_name, w, cap)
    try:
        rep = run_teacher_forced(m, SHAPES[shape_name], prompt, toks, logits)
        assert rep.steps == n_new
        # free-running generation matches too (identical tokens for fp32; for bf16 while
        # no near-tie has occurred)
        gen = m.generate(prompt, n_new)
        if SHAPES[shape_name].dtype == "f32":
            assert gen == toks
        else:
            assert gen[0] == toks[0] or rep.near_ties
    finally:
        m.close()


@pytest.mark.parametrize("shape_name,P,n_new,cap", [
    ("small_bf16", 100, 12, 160),
    ("hd128_bf16", 150, 12, 200),
    ("untied_bf16", 45, 12, 64),
])
def test_one_kernel_per_operation_path(monkeypatch, shape_name, P, n_new, cap):
    """bf16 decode steps as one kernel per operation (QW_MEGA=0) instead of the persistent
    decode-step kernel: the same parity."""
    monkeypatch.setenv("QW_MEGA", "0")
    w, prompt, toks, logits = oracle_run(shape_name, P, n_new)
    m = _model(shape_name, w, cap)
    try:
        assert m.decode_kernels_per_step() == 5 * SHAPES[shape_name].n_layers + 2
        rep = run_teacher_forced(m, SHAPES[shape_name], prompt, toks, logits)
        assert rep.steps == n_new
    finally:
        m.close()


def test_persistent_step_kernel_is_the_default_for_bf16():
    w, prompt, toks, logits = oracle_run("hd128_bf16", 150, 12)
    m = _model("hd128_bf16", w, 200)
    try:
        assert m.decode_kernels_per_step() == 1
    finally:
        m.close()
    wt, _, _, _ = oracle_run("tiny", 8, 8)
    m = _model("tiny", wt, 16)
    try:
        assert m.decode_kernels_per_step() == 5 * SHAPES["tiny"].n_layers + 2  # fp32: one per operation
    finally:
        m.close()


def test_tiny_without_graphs_matches(monkeypatch):
    monkeypatch.setenv("QW_NO_GRAPH", "1")
    w, prompt, toks, logits = oracle_run("tiny", 8, 8)
    m = _model("tiny", w, 16)
    try:
        run_teacher_forced(m, SHAPES["tiny"], prompt, toks, logits)
    finally:
        m.close()


@pytest.mark.parametrize("shape_name", ["small_bf16", "hd128_bf16", "gqa4_bf16", "gqa2_hd128_bf16"])
@pytest.mark.parametrize("simt,attn", [("0", "tc"), ("0", "mma"), ("0", "simt"), ("1", "tc")])
def test_bf16_prefill_paths(monkeypatch, shape_name, simt, attn):
    """The tensor-core prefill (default for bf16) with each of its attention kernels
    (QW_PREFILL_ATTN: tcgen05, mma.sync, CUDA cores) and the CUDA-core prefill
    (QW_PREFILL_SIMT=1) all match the oracle; 300 prompt tokens leave ragged query and
    key blocks, on head sizes 64 and 128 with odd and even query heads per KV head."""
    monkeypatch.setenv("QW_PREFILL_SIMT", simt)
    monkeypatch.setenv("QW_PREFILL_ATTN", attn)
    w, prompt, toks, logits = oracle_run(shape_name, 300, 4)
    m = _model(shape_name, w, 320)
    try:
        run_teacher_forced(m, SHAPES[shape_name], prompt, toks, logits)
    finally:
        m.close()


def test_0p5b_workload_full():
    wl = WORKLOADS["0p5b"]
    w, prompt, toks, logits = oracle_run(wl.shape, wl.prompt_len, wl.new_tokens)
    m = _model(wl.shape, w, wl.kv_capacity)
    try:
        rep = run_teacher_forced(m, SHAPES[wl.shape], prompt, toks, logits)
        assert rep.steps == wl.new_tokens
        record("0p5b 32-token prompt, 32 tokens", rep)
    finally:
        m.close()


def test_1p5b_workload_full():
    """The Qwen2.5-1.5B workload as the bench runs it: 128-token prompt, cache 2048, every
    one of the 100 tokens compared under teacher forcing."""
    wl = WORKLOADS["1p5b"]
    w, prompt, toks, logits = oracle_run(wl.shape, wl.prompt_len, wl.new_tokens)
    m = _model(wl.shape, w, wl.kv_capacity)
    try:
        rep = run_teacher_forced(m, SHAPES[wl.shape], prompt, toks, logits)
        assert rep.steps == wl.new_tokens
        record("1p5b 128-token prompt, 100 tokens", rep)
    finally:
        m.close()


def test_1p5b_long_context():
    """The long-context workload: a 4096-token prompt (tensor-core prefill at full size)
    into an 8192-position cache, then 32 of its 256 decode steps at 4096+ positions."""
    wl = WORKLOADS["1p5b_long"]
    w, prompt, toks, logits = oracle_run(wl.shape, wl.prompt_len, 33)
    m = _model(wl.shape, w, wl.kv_capacity)
    try:
        rep = run_teacher_forced(m, SHAPES[wl.shape], prompt, toks, logits)
        assert rep.steps == 33
        record("1p5b 4096-token prompt, 33 tokens", rep)
    finally:
        m.close()


def test_7b_shape_two_layers():
    """The Qwen2.5-Coder-7B shape (hidden 3584, 28/4 heads, MLP 18944, vocab 152064) on its
    first two layers: tensor-core prefill of a ragged 150-token prompt, then decode steps
    whose down projection runs K = 18944 through the GEMV's widest register tile."""
    w, prompt, toks, logits = oracle_run("7b_2l", 150, 6)
    m = _model("7b_2l", w, 200)
    try:
        rep = run_teacher_forced(m, SHAPES["7b_2l"], prompt, toks, logits)
        assert rep.steps == 6
        record("7b shape, 2 layers, 150-token prompt, 6 tokens", rep)
    finally:
        m.close()


def test_cuda_core_decode_attention(monkeypatch):
    """Decode attention on CUDA cores (QW_ATTN_MMA=0; the tensor-core kernel is the default)
    with its chunks merged in the o_proj GEMV, on a head_dim-128 shape."""
    monkeypatch.setenv("QW_ATTN_MMA", "0")
    w, prompt, toks, logits = oracle_run("hd128_bf16", 150, 12)
    m = _model("hd128_bf16", w, 200)
    try:
        run_teacher_forced(m, SHAPES["hd128_bf16"], prompt, toks, logits)
    finally:
        m.close()


# ---- edge cases ----------------------------------------------------------------------

def test_single_token_prompt_and_full_capacity():
    s = SHAPES["tiny"]
    w = make_weights(s)
    prompt = make_prompt(s, 1)
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w)
    toks, logits = oracle.generate(om, prompt, 16)   # 1 + 15 positions = capacity 16
    m = _model("tiny", w, 16)
    try:
        run_teacher_forced(m, s, prompt, toks, logits)
        assert m.position() == 16
        from qwen2_decoder_forward_decode_gb300 import QwError
        with pytest.raises(QwError) as e:
            m.decode_step()
        assert e.value.status == 3  # QW_ERR_CAPACITY
    finally:
        m.close()


def test_prompt_equal_to_capacity_and_over():
    s = SHAPES["tiny"]
    w = make_weights(s)
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w)
    prompt = make_prompt(s, 16)
    toks, logits = oracle.generate(om, prompt, 1)
    m = _model("tiny", w, 16)
    from qwen2_decoder_forward_decode_gb300 import QwError
    try:
        rep = StepReport()
        t = m.prefill(prompt)
        check_step(s, m.logits(), t, logits[0], toks[0], rep)
        with pytest.raises(QwError) as e:
            m.prefill(make_prompt(s, 17))
        assert e.value.status == 3
        with pytest.raises(QwError) as e:
            m.generate(make_prompt(s, 10), 8)   # 10 + 8 - 1 > 16
        assert e.value.status == 3
    finally:
        m.close()


def test_bad_tokens_rejected():
    s = SHAPES["tiny"]
    w = make_weights(s)
    m = _model("tiny", w, 16)
    from qwen2_decoder_forward_decode_gb300 import QwError
    try:
        with pytest.raises(QwError) as e:
            m.prefill(np.array([1, 2, 256], dtype=np.int32))
        assert e.value.status == 4
        with pytest.raises(QwError) as e:
            m.prefill(np.array([], dtype=np.int32))   # empty prompt
        assert e.value.status == 1
        with pytest.raises(QwError) as e:
            m.prefill(np.array([1], dtype=np.int32), seq=1)   # the model holds one sequence
        assert e.value.status == 1
        with pytest.raises(QwError) as e:
            m.generate(np.array([1, 2], dtype=np.int32), 0)   # max_new counts the first token
        assert e.value.status == 1
        with pytest.raises(QwError) as e:
            m.decode_step()   # nothing prefilled
        assert e.value.status == 1
        m.prefill(np.array([1, 2, 3], dtype=np.int32))
        with pytest.raises(QwError) as e:
            m.decode_step(feed=[-1])
        assert e.value.status == 4
        m.decode_step(feed=[5])   # still usable
    finally:
        m.close()


def test_stop_set_ends_generation_like_the_oracle():
    """qw_generate_stops: the first produced token in the stop set ends the run, as in the
    oracle's generate with eos_ids; a set without produced ids runs to max_new."""
    s = SHAPES["tiny"]
    w = make_weights(s)
    prompt = make_prompt(s, 5)
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w)
    toks, _ = oracle.generate(om, prompt, 12)
    absent = next(v for v in range(s.vocab) if v not in toks)
    stops = [absent, toks[6], toks[4]]
    want, _ = oracle.generate(om, prompt, 12, eos_ids=stops)
    m = _model("tiny", w, 20)
    try:
        assert m.generate(prompt, 12, eos_ids=stops) == want
        assert m.position() == len(prompt) + len(want) - 1
        assert m.generate(prompt, 12, eos_ids=[absent]) == toks
        assert m.generate(prompt, 12, eos_ids=[]) == toks
    finally:
        m.close()


def test_eos_stops_generation_and_keeps_state():
    s = SHAPES["tiny"]
    w = make_weights(s)
    prompt = make_prompt(s, 5)
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w)
    toks, _ = oracle.generate(om, prompt, 10)
    eos = toks[3]
    want, _ = oracle.generate(om, prompt, 10, eos=eos)
    m = _model("tiny", w, 16)
    try:
        got = m.generate(prompt, 10, eos=eos)
        assert got == want
        assert m.position() == len(prompt) + len(want) - 1
        # continuing after the stop equals the oracle continuing the same sequence
        nxt = int(m.decode_step()[0])
        assert nxt == oracle.generate(om, list(prompt) + want, 1)[0][0]
    finally:
        m.close()


def test_decode_is_deterministic():
    wl = WORKLOADS["0p5b"]
    w, prompt, toks, logits = oracle_run(wl.shape, wl.prompt_len, wl.new_tokens)
    m = _model(wl.shape, w, wl.kv_capacity)
    try:
        a = m.generate(prompt, 8)
        za = m.logits()
        b = m.generate(prompt, 8)
        zb = m.logits()
        assert a == b
        np.testing.assert_array_equal(za, zb)
    finally:
        m.close()


@pytest.mark.parametrize("P", [128, 600])
def test_prefill_is_deterministic(P):
    """Two prefills of the same prompt give bit-identical logits and token: the tensor-core
    chain (split-K GEMMs at 128 tokens, CTA-pair GEMMs at 600, the tcgen05 attention,
    programmatic dependent launch between every kernel) reduces in a fixed order and adds no
    floats atomically."""
    s = SHAPES["1p5b"]
    w = make_weights(s)
    prompt = make_prompt(s, P)
    m = _model("1p5b", w, P + 8)
    try:
        ta = m.prefill(prompt)
        za = np.array(m.logits(), copy=True)
        m.reset()
        tb = m.prefill(prompt)
        zb = np.array(m.logits(), copy=True)
        assert ta == tb
        np.testing.assert_array_equal(za, zb)
    finally:
        m.close()


def test_fault_injection_at_decode_leaves_the_model_usable(monkeypatch):
    """QW_FAULT=launch fails a decode call with QW_ERR_FAULT_INJECTED before any launch;
    the sequence keeps its length and the next call continues it exactly."""
    from qwen2_decoder_forward_decode_gb300 import QwError
    w, prompt, toks, logits = oracle_run("tiny", 8, 8)
    m = _model("tiny", w, 16)
    try:
        m.prefill(prompt)
        monkeypatch.setenv("QW_FAULT", "launch")
        with pytest.raises(QwError) as e:
            m.decode_step(feed=[toks[0]])
        assert e.value.status == 7
        assert m.position() == len(prompt)
        monkeypatch.delenv("QW_FAULT")
        rep = StepReport()
        t = int(m.decode_step(feed=[toks[0]])[0])
        check_step(SHAPES["tiny"], m.logits(), t, logits[1], toks[1], rep, "after the injected fault")
    finally:
        m.close()


def test_reset_clears_the_last_error():
    from qwen2_decoder_forward_decode_gb300 import QwError, lib
    w, prompt, _, _ = oracle_run("tiny", 8, 8)
    m = _model("tiny", w, 16)
    try:
        m.prefill(prompt)
        with pytest.raises(QwError):
            m.decode_step(feed=[-5])
        assert lib().qw_last_error().decode()
        m.reset(0)
        assert lib().qw_last_error().decode() == ""
        assert m.position() == 0
    finally:
        m.close()


def _overflowing_weights(shape_name):
    """The shape's weights with layer 0's value bias at 70144 (a bf16 value above the fp16
    maximum 65504): every value written to the fp16 KV cache of layer 0 overflows."""
    from synth import round_to_bf16
    s = SHAPES[shape_name]
    w = dict(make_weights(s))
    b = np.full(s.n_kv_heads * s.head_dim, 70000.0, dtype=np.float32)
    w["model.layers.0.self_attn.v_proj.bias"] = round_to_bf16(b)
    assert float(w["model.layers.0.self_attn.v_proj.bias"][0]) == 70144.0
    return s, w


@pytest.mark.parametrize("max_seqs", [1, 2])
def test_fp16_overflow_is_reported(max_seqs):
    """A value beyond the fp16 range written to the KV cache is an error (QW_ERR_NUMERIC),
    reported by the prefill and by decode steps (single-sequence and batched), never a
    silent infinity."""
    from qwen2_decoder_forward_decode_gb300 import QwError
    s, w = _overflowing_weights("small_bf16")
    m = _model("small_bf16", w, 64, max_seqs=max_seqs)
    try:
        for b in range(max_seqs):
            with pytest.raises(QwError) as e:
                m.prefill(make_prompt(s, 10 + b), seq=b)
            assert e.value.status == 8
        with pytest.raises(QwError) as e:
            m.decode_step(feed=np.ones(max_seqs, dtype=np.int32))
        assert e.value.status == 8
    finally:
        m.close()
