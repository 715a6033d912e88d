"""Seeded synthetic weights and token ids.

Recipe (the same for every consumer):
  * every weight matrix, embedding and bias is N(0, 0.02); RMSNorm gains are
    1 + N(0, 0.02) (unit gains, perturbed so that a dropped gain multiply shows);
  * tensor ``index`` (its position in ``tensor_shapes``) is drawn flat, in blocks of
    2^22 values; block c draws from its own stream ``default_rng([seed, index, c])``, so
    any subset can be regenerated alone and blocks are drawn in parallel;
  * bf16 shapes round every value to bf16 (round-to-nearest-even) and keep it as the
    exactly representable float32 value; f32 shapes keep the float32 draw;
  * prompt ids are uniform on [0, vocab) from ``default_rng(1)``; batched prompt
    lengths are ``default_rng(2).integers(lo, hi + 1, n)`` and sequence b's ids come
    from ``default_rng(3 + b)``.

Tensor names follow the Hugging Face / safetensors layout used by the pages
("LLM Speedrun: Architecture", Implementing Qwen / Harness: model.layers.{i}.self_attn.
q_proj.weight and so on). Matrices are row-major [out, in].
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .shapes import Shape

WEIGHT_STD = 0.02


def tensor_shapes(s: Shape):
    """Ordered (name, shape, kind) for every parameter tensor of shape ``s``.

    kind is "mat" (N(0, 0.02)) or "gain" (1 + N(0, 0.02)).
    """
    H, I, V = s.hidden, s.intermediate, s.vocab
    q_out = s.n_heads * s.head_dim
    kv_out = s.n_kv_heads * s.head_dim
    out = [("model.embed_tokens.weight", (V, H), "mat")]
    for i in range(s.n_layers):
        p = f"model.layers.{i}."
        out += [
            (p + "input_layernorm.weight", (H,), "gain"),
            (p + "self_attn.q_proj.weight", (q_out, H), "mat"),
            (p + "self_attn.k_proj.weight", (kv_out, H), "mat"),
            (p + "self_attn.v_proj.weight", (kv_out, H), "mat"),
        ]
        if s.qkv_bias:
            out += [
                (p + "self_attn.q_proj.bias", (q_out,), "mat"),
                (p + "self_attn.k_proj.bias", (kv_out,), "mat"),
                (p + "self_attn.v_proj.bias", (kv_out,), "mat"),
            ]
        out += [
            (p + "self_attn.o_proj.weight", (H, q_out), "mat"),
            (p + "post_attention_layernorm.weight", (H,), "gain"),
            (p + "mlp.gate_proj.weight", (I, H), "mat"),
            (p + "mlp.up_proj.weight", (I, H), "mat"),
            (p + "mlp.down_proj.weight", (H, I), "mat"),
        ]
    out.append(("model.norm.weight", (H,), "gain"))
    if not s.tied:
        out.append(("lm_head.weight", (V, H), "mat"))
    return out


def tensor_names(s: Shape):
    return [n for n, _, _ in tensor_shapes(s)]


def param_count(s: Shape) -> int:
    total = 0
    for _, shp, _ in tensor_shapes(s):
        n = 1
        for d in shp:
            n *= d
        total += n
    return total


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    r &= np.uint32(0xFFFF0000)
    return r.view(np.float32).reshape(a.shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already exactly bf16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


BLOCK = 1 << 22


def _fill_block(out_flat, seed, index, c, kind, bf16):
    lo = c * BLOCK
    hi = min(out_flat.size, lo + BLOCK)
    rng = np.random.default_rng([seed, index, c])
    a = rng.standard_normal(size=hi - lo, dtype=np.float32)
    a *= np.float32(WEIGHT_STD)
    if kind == "gain":
        a += np.float32(1.0)
    if bf16:
        a = round_to_bf16(a)
    out_flat[lo:hi] = a


def make_weights(s: Shape, seed: int = 0, layers=None, threads: int = None):
    """Return {name: float32 ndarray}. ``layers`` limits the per-layer tensors drawn
    (None = all); the global tensors are always drawn."""
    import os
    bf16 = s.dtype == "bf16"
    out, jobs = {}, []
    for idx, (name, shp, kind) in enumerate(tensor_shapes(s)):
        if layers is not None and name.startswith("model.layers."):
            li = int(name.split(".")[2])
            if li not in layers:
                continue
        arr = np.empty(shp, dtype=np.float32)
        out[name] = arr
        flat = arr.reshape(-1)
        for c in range((flat.size + BLOCK - 1) // BLOCK):
            jobs.append((flat, idx, c, kind))
    n = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(lambda j: _fill_block(j[0], seed, j[1], j[2], j[3], bf16), jobs))
    return out


def make_prompt(s: Shape, n: int, seed: int = 1) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, s.vocab, n).astype(np.int32)


def make_batch_prompts(s: Shape, n_seqs: int, lo: int, hi: int):
    lens = np.random.default_rng(2).integers(lo, hi + 1, n_seqs)
    return [np.random.default_rng(3 + b).integers(0, s.vocab, int(L)).astype(np.int32)
            for b, L in enumerate(lens)]
