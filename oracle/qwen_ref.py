"""Plain CPU oracle of the Qwen2 decoder forward pass, in float64.

(A float32 mode, ``OracleModel(..., dtype=np.float32)``, runs the same steps in the precision
of [LSA]'s numpy model code, whose arrays are all float32. It only serves as the timed CPU
baseline; parity always uses float64.)

TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the bench's
CPU-baseline / reference legs may import this module. It shares no code with the CUDA
library: the only thing both sides use is the seeded input generator in ``synth``.

Sources (page title, then the section on it):
  [LSA]  "LLM Speedrun: Architecture" - Transformer architecture (attention, causal mask,
         SwiGLU FFN, pre-norm residuals, GQA, RoPE, Decoding / LM head / KV cache) and
         Implementing Qwen (bias, split-half RoPE, the Qwen model code).
  [AUG]  "augur" - Features (RMSNorm placement, RoPE on q and k, GQA, causal masking,
         SwiGLU MLP, decoder block order, greedy generation, EOS stop, prefill/decode
         split, preallocated KV cache).
  [QIE]  "Building a Qwen2.5-1.5B Inference Engine From Scratch" - §1 (prefill vs
         decode), §1.1 (reference run without a cache, first-token logits).

Notation follows [LSA]: activations are column matrices [features, T] ("all vectors
are column vectors"); weights are [out, in] so a projection is ``W @ x``.

Readings where the pages are garbled or silent:
  * RoPE frequency of pair i is theta^(-2i/head_dim), i < head_dim/2; pairs are
    (i, i + head_dim/2) ("split-half"); angle = position * frequency in float64.
  * RoPE is applied to q and k after the bias and before k enters the cache; v is not
    rotated.
  * Score scale is 1/sqrt(d_k) with d_k = hidden / n_heads (= head_dim here).
  * Query head h reads KV head floor(h / (n_heads / n_kv_heads)).
  * Masked scores are set to -1e9 as on [LSA]; keys at positions > the query's own
    position are masked (at least one key, the query's own, is always open).
  * eps sits inside the square root of the RMSNorm; the gain multiplies afterwards.
  * Only the last position gets the final norm and the LM head; the LM head is the
    embedding matrix (tied) unless an untied one is given.
  * Greedy argmax takes the lowest index among equal maxima.
"""
import math
from dataclasses import dataclass

import numpy as np

MASK_VALUE = -1e9


@dataclass
class OracleConfig:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    tied: bool = True

    @staticmethod
    def from_shape(s):
        return OracleConfig(s.n_layers, s.hidden, s.n_heads, s.n_kv_heads, s.head_dim,
                            s.intermediate, s.vocab, s.rms_eps, s.rope_theta, s.tied)


class OracleModel:
    """Weights held as float64 copies of the given arrays (bf16 values are exact in f64),
    or float32 copies with dtype=np.float32 (every activation then stays float32)."""

    def __init__(self, cfg: OracleConfig, weights: dict, dtype=np.float64):
        self.cfg = cfg
        self.dtype = np.dtype(dtype)
        self.w = {k: np.asarray(v, dtype=self.dtype) for k, v in weights.items()}

    def layer(self, i, name):
        return self.w.get(f"model.layers.{i}.{name}")

    @property
    def lm_head(self):
        if self.cfg.tied:
            return self.w["model.embed_tokens.weight"]
        return self.w["lm_head.weight"]


# --- building blocks -----------------------------------------------------------------

def embed(E, token_ids):
    """Token embedding [AUG Features "Full forward pass"; LSA "Setting up the inputs"]:
    column t of the result is row token_ids[t] of E [V, H]."""
    ids = np.asarray(token_ids, dtype=np.int64)
    if ids.min() < 0 or ids.max() >= E.shape[0]:
        raise ValueError("token id outside the vocabulary")
    return np.ascontiguousarray(E[ids, :].T)


def rms_norm(x, gain, eps):
    """RMSNorm over the feature axis [LSA Normalization; AUG RMSNorm]:
    x / sqrt(mean(x^2) + eps), then times the gain."""
    mean_sq = np.mean(x * x, axis=0, keepdims=True)
    return (x / np.sqrt(mean_sq + eps)) * gain[:, None]


def rope_frequencies(head_dim, theta):
    """Rotation frequency of pair i: theta^(-2i/head_dim) [LSA RoPE, decaying frequencies]."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_rotate(x, positions, theta):
    """Split-half rotary embedding of one head [LSA Split-half RoPE implementation].

    x is [head_dim, T]; element i (first half) and element i + head_dim/2 (second half)
    form one complex number (real, imaginary) rotated by positions[t] * freq_i.
    """
    hd = x.shape[0]
    half = hd // 2
    ang = np.outer(rope_frequencies(hd, theta), np.asarray(positions, dtype=np.float64))
    c, s = np.cos(ang).astype(x.dtype, copy=False), np.sin(ang).astype(x.dtype, copy=False)  # (f32 mode)
    re, im = x[:half], x[half:]
    out = np.empty_like(x)
    out[:half] = re * c - im * s
    out[half:] = im * c + re * s
    return out


def softmax_rows(s):
    """Softmax along the last axis with the maximum subtracted first [LSA softmax]."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def silu(x):
    """Swish / SiLU: x / (1 + e^-x) [LSA SwiGLU FFN]."""
    return x / (1.0 + np.exp(-x))


def attend_one_head(q, K, V, q_positions, d_k):
    """Causal scaled dot-product attention of one query head over one KV head
    [LSA Attention, Causal mask, Softmax].

    q: [hd, T] rotated queries at absolute positions q_positions; K, V: [hd, Ttot] keys
    (rotated) and values for positions 0..Ttot-1. Returns [hd, T].
    """
    scores = (q.T @ K) / math.sqrt(d_k)                    # [T, Ttot] (a Python float keeps f32 mode f32)
    key_pos = np.arange(K.shape[1])
    masked = key_pos[None, :] > np.asarray(q_positions)[:, None]
    scores = np.where(masked, MASK_VALUE, scores)
    p = softmax_rows(scores)
    return V @ p.T


class KVCache:
    """Per-layer keys and values, [n_kv_heads, head_dim, T], grown along T
    [LSA Decoding / KV cache; AUG Preallocated KV-cache]."""

    def __init__(self, n_layers):
        self.k = [None] * n_layers
        self.v = [None] * n_layers

    def append(self, layer, k, v):
        if self.k[layer] is None:
            self.k[layer], self.v[layer] = k, v
        else:
            self.k[layer] = np.concatenate([self.k[layer], k], axis=2)
            self.v[layer] = np.concatenate([self.v[layer], v], axis=2)
        return self.k[layer], self.v[layer]

    @property
    def length(self):
        return 0 if self.k[0] is None else self.k[0].shape[2]


def attention_block(m: OracleModel, li, xn, positions, cache: KVCache):
    """Grouped-query attention of layer li on normalised input xn [H, T]
    [LSA GQA, Introducing bias; AUG Grouped-query attention]."""
    c = m.cfg
    T = xn.shape[1]
    hd, nq, nkv = c.head_dim, c.n_heads, c.n_kv_heads
    group = nq // nkv

    def proj(name):
        y = m.layer(li, f"self_attn.{name}.weight") @ xn
        b = m.layer(li, f"self_attn.{name}.bias")
        return y if b is None else y + b[:, None]

    q = proj("q_proj").reshape(nq, hd, T)
    k = proj("k_proj").reshape(nkv, hd, T)
    v = proj("v_proj").reshape(nkv, hd, T)
    q = np.stack([rope_rotate(q[h], positions, c.rope_theta) for h in range(nq)])
    k = np.stack([rope_rotate(k[h], positions, c.rope_theta) for h in range(nkv)])
    K, V = cache.append(li, k, v)
    d_k = c.hidden // nq
    heads = [attend_one_head(q[h], K[h // group], V[h // group], positions, d_k)
             for h in range(nq)]
    o = np.concatenate(heads, axis=0)                       # [nq*hd, T]
    return m.layer(li, "self_attn.o_proj.weight") @ o


def mlp_block(m: OracleModel, li, xn):
    """SwiGLU MLP: down(up(x) * silu(gate(x))) [LSA SwiGLU FFN; AUG Qwen MLP]."""
    gate = m.layer(li, "mlp.gate_proj.weight") @ xn
    up = m.layer(li, "mlp.up_proj.weight") @ xn
    return m.layer(li, "mlp.down_proj.weight") @ (up * silu(gate))


def decoder_layer(m: OracleModel, li, x, positions, cache):
    """Pre-norm block: h = x + attn(norm1(x)); out = h + mlp(norm2(h))
    [LSA Why pre-norm over post-norm, Summed up; AUG Decoder blocks]."""
    eps = m.cfg.rms_eps
    h = x + attention_block(m, li, rms_norm(x, m.layer(li, "input_layernorm.weight"), eps),
                            positions, cache)
    return h + mlp_block(m, li, rms_norm(h, m.layer(li, "post_attention_layernorm.weight"),
                                         eps))


def forward_hidden(m: OracleModel, token_ids, positions, cache):
    """All layers on the given tokens; returns the residual stream [H, T]."""
    x = embed(m.w["model.embed_tokens.weight"], token_ids)
    for li in range(m.cfg.n_layers):
        x = decoder_layer(m, li, x, positions, cache)
    return x


def final_logits(m: OracleModel, x_last):
    """Final RMSNorm of the last position and the LM head [LSA Transformer output,
    Decoding; AUG Full forward pass]. x_last: [H]. Returns logits [V]."""
    h = rms_norm(x_last[:, None], m.w["model.norm.weight"], m.cfg.rms_eps)[:, 0]
    return m.lm_head @ h


def greedy(z):
    """Greedy choice: index of the largest logit, lowest index on ties [AUG Greedy
    generation]. Non-finite logits are an error."""
    if not np.all(np.isfinite(z)):
        raise FloatingPointError("non-finite logits")
    return int(np.argmax(z))


def step(m: OracleModel, token_ids, positions, cache):
    """One forward step (prefill of several tokens, or decode of one): returns
    (next_token, logits of the last position)."""
    x = forward_hidden(m, token_ids, positions, cache)
    z = final_logits(m, x[:, -1])
    return greedy(z), z


def _is_stop(t, eos, eos_ids):
    return (eos >= 0 and t == eos) or (eos_ids is not None and t in eos_ids)


def generate(m: OracleModel, prompt, max_new, eos=-1, feed=None, eos_ids=None):
    """Greedy generation with a KV cache [AUG Prefill/decode split, EOS stopping].

    Step 0 runs the whole prompt at positions 0..P-1; each later step runs the last
    token alone at position len-1. ``max_new`` counts every generated token, the
    prefill's included. With ``feed`` (teacher forcing) the token run at decode step i
    is feed[i-1] instead of the previous argmax. A token equal to ``eos``, or to any id
    of the set ``eos_ids`` ([LSA] Implementing Qwen: generate_tokens and its eos_ids), is
    appended, then generation stops. Returns (tokens, [logits per step]).
    """
    eos_ids = None if eos_ids is None else {int(e) for e in eos_ids}
    cache = KVCache(m.cfg.n_layers)
    seq = [int(t) for t in prompt]
    out, logits = [], []
    for i in range(max_new):
        if i == 0:
            t, z = step(m, seq, np.arange(len(seq)), cache)
        else:
            last = seq[-1] if feed is None else int(feed[i - 1])
            if feed is not None:
                seq[-1] = last
            t, z = step(m, [last], np.array([len(seq) - 1]), cache)
        out.append(t)
        logits.append(z)
        seq.append(t)
        if _is_stop(t, eos, eos_ids):
            break
    return out, logits


def generate_uncached(m: OracleModel, prompt, max_new, eos=-1, feed=None):
    """The same generation recomputing the whole sequence every step with a fresh cache
    (the cache-free reference run of [QIE] §1.1)."""
    seq = [int(t) for t in prompt]
    out, logits = [], []
    for i in range(max_new):
        if i > 0 and feed is not None:
            seq[-1] = int(feed[i - 1])
        t, z = step(m, seq, np.arange(len(seq)), KVCache(m.cfg.n_layers))
        out.append(t)
        logits.append(z)
        seq.append(t)
        if eos >= 0 and t == eos:
            break
    return out, logits
