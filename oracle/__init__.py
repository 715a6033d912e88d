"""CPU oracle of the Qwen2 decoder forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline and
reference legs may import this package; the library never does.
"""
from .qwen_ref import (  # noqa: F401
    OracleConfig, OracleModel, KVCache, embed, rms_norm, rope_frequencies, rope_rotate,
    softmax_rows, silu, attend_one_head, attention_block, mlp_block, decoder_layer,
    forward_hidden, final_logits, greedy, step, generate, generate_uncached, MASK_VALUE,
)
