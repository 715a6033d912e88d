"""Several independent sequences in one model (max_seqs > 1): each sequence gives the
result of running it alone, and the oracle's result, under teacher forcing."""
import numpy as np
import pytest

import oracle
from parity import StepReport, check_step
from synth import SHAPES, make_batch_prompts, make_weights

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("shape_name", ["small_f32", "small_bf16"])
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
