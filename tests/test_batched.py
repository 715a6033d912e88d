"""Several independent sequences in one model (max_seqs > 1): each sequence gives the
result of running it alone, and the oracle's result, under teacher forcing."""
import numpy as np
import pytest

import oracle
from parity import StepReport, check_step, record, shape_weights
from synth import SHAPES, WORKLOADS, make_batch_prompts, make_weights

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("shape_name", ["small_f32", "small_bf16", "untied_bf16"])
def test_batched_sequences_match_oracle(shape_name):
    from qwen2_decoder_forward_decode_gb300 import DeviceWeights, Model
    s = SHAPES[shape_name]
    w = make_weights(s)
    prompts = make_batch_prompts(s, 4, 5, 40)
    n_new = 6
    om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w)
    refs = [oracle.generate(om, p, n_new) for p in prompts]
    m = Model(s, DeviceWeights(w, 1 if s.dtype == "bf16" else 0), 64, max_seqs=4)
    rep = StepReport()
    try:
        for b, p in enumerate(prompts):
            t = m.prefill(p, seq=b)
            check_step(s, m.logits(b), t, refs[b][1][0], refs[b][0][0], rep, f"seq {b} prefill")
        for i in range(1, n_new):
            feed = np.array([refs[b][0][i - 1] for b in range(4)], dtype=np.int32)
            toks = m.decode_step(feed=feed)
            for b in range(4):
                check_step(s, m.logits(b), int(toks[b]), refs[b][1][i], refs[b][0][i], rep,
                           f"seq {b} step {i}")
        for b, p in enumerate(prompts):
            assert m.position(b) == len(p) + n_new - 1
    finally:
        m.close()


def _run_batch(s, w, prompts, n_new, cap, check_seqs, reset_at=None, reset_seq=None, om=None):
    """Prefill every prompt into its own sequence slot, then decode all slots together,
    feeding the oracle's tokens to the sequences in check_seqs (compared every step) and
    the device's own tokens to the others."""
    from qwen2_decoder_forward_decode_gb300 import DeviceWeights, Model
    if om is None:
        om = oracle.OracleModel(oracle.OracleConfig.from_shape(s), w)
    refs = {b: oracle.generate(om, prompts[b], n_new) for b in check_seqs}
    S = len(prompts)
    m = Model(s, DeviceWeights(w, 1), cap, max_seqs=S)
    rep = StepReport()
    try:
        last = np.zeros(S, dtype=np.int32)
        for b, p in enumerate(prompts):
            last[b] = m.prefill(p, seq=b)
            if b in refs:
                check_step(s, m.logits(b), int(last[b]), refs[b][1][0], refs[b][0][0], rep, f"seq {b} prefill")
        live = set(range(S))
        for i in range(1, n_new):
            if reset_at is not None and i == reset_at:
                m.reset(reset_seq)
                live.discard(reset_seq)
            feed = np.array([refs[b][0][i - 1] if b in refs else last[b] for b in range(S)], dtype=np.int32)
            toks = m.decode_step(feed=feed)
            for b in live:
                last[b] = toks[b]
                if b in refs:
                    check_step(s, m.logits(b), int(toks[b]), refs[b][1][i], refs[b][0][i], rep,
                               f"seq {b} step {i}")
        for b in live:
            assert m.position(b) == len(prompts[b]) + n_new - 1
        if reset_seq is not None:
            assert m.position(reset_seq) == 0
    finally:
        m.close()
    return rep


def test_batched_16_sequences_match_oracle():
    """16 sequences of ragged lengths decoded together (weights read once per step for all
    of them): every sequence matches the oracle at every step; a sequence reset midway
    leaves the batch and the others continue unchanged."""
    s = SHAPES["hd128_bf16"]
    w = make_weights(s)
    prompts = make_batch_prompts(s, 16, 5, 60)
    rep = _run_batch(s, w, prompts, 5, 96, set(range(16)) - {9}, reset_at=3, reset_seq=9)
    record("hd128 batched, 16 ragged sequences", rep)


def test_batched_1p5b_workload():
    """The batched workload at its own configuration: 16 sequences of the Qwen2.5-1.5B
    shape with prompts of 256-2048 tokens (the workload's seeds), a 2304-position cache per
    sequence, all 16 decoding together. Four of them (the longest and shortest prompts and
    two others) follow the oracle's tokens and are compared at every one of 17 steps (the
    prefill and 16 decode steps) at the chunk sizes the bench runs; the other twelve run
    their own tokens."""
    wl = WORKLOADS["1p5b_batch"]
    s = SHAPES[wl.shape]
    w, om = shape_weights(wl.shape)
    prompts = make_batch_prompts(s, wl.n_seqs, *wl.batch_len_range)
    lens = [len(p) for p in prompts]
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    check = {longest, shortest} | {b for b in (3, 11) if b not in (longest, shortest)}
    assert len(check) >= 4
    rep = _run_batch(s, w, prompts, 17, wl.kv_capacity, check, om=om)
    assert rep.steps == 17 * len(check)
    record(f"1p5b batched, 16 sequences ({min(lens)}-{max(lens)} tokens), {len(check)} compared", rep)


def test_batched_1p5b_shape_small_prompts():
    """The Qwen2.5-1.5B shape with 8 short sequences decoded together; two of them are
    compared with the oracle at every step."""
    s = SHAPES[WORKLOADS["1p5b_batch"].shape]
    w, om = shape_weights("1p5b")
    prompts = make_batch_prompts(s, 8, 8, 40)
    rep = _run_batch(s, w, prompts, 4, 64, {0, 5}, om=om)
    record("1p5b batched, 8 short sequences", rep)


@pytest.mark.parametrize("env", [{"QW_BATCHED_ATTN_MMA": "0"}, {"QW_BATCHED_SPLITS": "1"}])
def test_batched_alternative_kernels(monkeypatch, env):
    """The CUDA-core batched attention (off by default), and the tensor-core one with a
    single chunk per sequence (contexts of 65+ positions then span two 64-position tiles),
    match the oracle on 16 ragged sequences."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    s = SHAPES["hd128_bf16"]
    w = make_weights(s)
    prompts = make_batch_prompts(s, 16, 40, 120)
    _run_batch(s, w, prompts, 4, 128, {0, 7, 15})
