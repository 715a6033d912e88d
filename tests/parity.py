"""Shared helpers for comparing the CUDA path with the CPU oracle."""
import numpy as np

import oracle
from synth import SHAPES, make_weights, make_prompt

FP32_TOL = 1e-4      # max |logit difference| for fp32 models
BF16_REL_TOL = 2e-2  # max |logit difference| / std(oracle logits) for bf16 models


class StepReport:
    def __init__(self):
        self.near_ties = 0
        self.max_err = 0.0
        self.max_rel = 0.0
        self.steps = 0


def check_step(shape, z_gpu, tok_gpu, z_ref, tok_ref, rep: StepReport, where=""):
    """Acceptance rule for one step.

    fp32: identical token, max |dz| <= 1e-4.
    bf16: max |dz| <= 2e-2 * std(z_ref); the GPU token equals the oracle's wherever the
    oracle's top-1/top-2 gap exceeds twice that band, and otherwise lies inside the band
    below the oracle's maximum (those steps are counted as near-ties).
    In both cases the GPU token is the lowest index of the GPU logits' maximum."""
    z_gpu = np.asarray(z_gpu, dtype=np.float64)
    assert np.all(np.isfinite(z_gpu)), f"{where}: non-finite logits"
    own = int(np.argmax(z_gpu))
    assert tok_gpu == own, f"{where}: device argmax {tok_gpu} != argmax of its logits {own}"
    err = float(np.max(np.abs(z_gpu - z_ref)))
    rep.steps += 1
    rep.max_err = max(rep.max_err, err)
    if shape.dtype == "f32":
        assert tok_gpu == tok_ref, f"{where}: token {tok_gpu} != oracle {tok_ref}"
        assert err <= FP32_TOL, f"{where}: max|dz| {err:.3e} > {FP32_TOL}"
        return
    tol = BF16_REL_TOL * float(np.std(z_ref))
    rep.max_rel = max(rep.max_rel, err / float(np.std(z_ref)))
    assert err <= tol, f"{where}: max|dz| {err:.4f} > 2e-2*std {tol:.4f}"
    top2 = np.partition(z_ref, -2)[-2:]
    gap = float(top2[1] - top2[0])
    if gap > 2 * tol:
        assert tok_gpu == tok_ref, f"{where}: token {tok_gpu} != oracle {tok_ref} (gap {gap:.4f})"
    else:
        rep.near_ties += 1
        assert z_ref[tok_gpu] >= z_ref.max() - tol, f"{where}: near-tie token outside the band"


def run_teacher_forced(model, shape, prompt, ref_toks, ref_logits, seq=0):
    """Prefill then decode feeding the oracle's tokens; compare every step."""
    rep = StepReport()
    t = model.prefill(prompt, seq=seq)
    check_step(shape, model.logits(seq), t, ref_logits[0], ref_toks[0], rep, "prefill")
    for i in range(1, len(ref_toks)):
        feed = np.zeros(model.max_seqs, dtype=np.int32)
        feed[seq] = ref_toks[i - 1]
        t = int(model.decode_step(feed=feed)[seq])
        check_step(shape, model.logits(seq), t, ref_logits[i], ref_toks[i], rep, f"decode {i}")
    return rep


_weight_cache = {}
_oracle_cache = {}

# (test, steps compared, near-tie steps, max |dz| / std) of every parity run, printed in the
# session summary (tests/conftest.py)
REPORTS = []


def record(name, rep: StepReport):
    REPORTS.append((name, rep.steps, rep.near_ties, rep.max_rel if rep.max_rel else rep.max_err))


def shape_weights(shape_name):
    """(float32 weights, float64 oracle model) of a shape, drawn once per session."""
    if shape_name not in _weight_cache:
        s = SHAPES[shape_name]
        w = make_weights(s)
        _weight_cache[shape_name] = (w, oracle.OracleModel(oracle.OracleConfig.from_shape(s), w))
    return _weight_cache[shape_name]


def oracle_run(shape_name, prompt_len, n_new, seed_prompt=1):
    key = (shape_name, prompt_len, n_new, seed_prompt)
    if key not in _oracle_cache:
        s = SHAPES[shape_name]
        w, om = shape_weights(shape_name)
        prompt = make_prompt(s, prompt_len, seed=seed_prompt)
        toks, logits = oracle.generate(om, prompt, n_new)
        _oracle_cache[key] = (w, prompt, toks, logits)
    return _oracle_cache[key]
