"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a value printed on a
page, a closed form, an invariant the pages state, a special case that reduces to a
library routine, or brute force on a tiny input. None needs a GPU.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import OracleConfig, OracleModel
from synth import SHAPES, make_weights, make_prompt, param_count, round_to_bf16, tensor_names

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_model(shape="tiny", seed=0, **over):
    s = SHAPES[shape]
    w = make_weights(s, seed=seed)
    cfg = OracleConfig.from_shape(s)
    for k, v in over.items():
        setattr(cfg, k, v)
    return OracleModel(cfg, w), w, s


# --- parameter count (page value) -------------------------------------------------------

def test_param_count_matches_page():
    # "Building a Qwen2.5-1.5B Inference Engine From Scratch", §1.1
    with open(os.path.join(GOLDEN, "param_count.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert rows == [["1p5b", "1543714304"]]
    assert param_count(SHAPES["1p5b"]) == 1543714304


def test_oracle_reads_every_tensor_and_only_those():
    m, w, s = tiny_model()
    seen = set()

    class Tracking(dict):
        def __getitem__(self, k):
            seen.add(k)
            return dict.__getitem__(self, k)

        def get(self, k, d=None):
            if k in self:
                seen.add(k)
            return dict.get(self, k, d)

    m.w = Tracking(m.w)
    oracle.generate(m, make_prompt(s, 3), 2)
    assert seen == set(tensor_names(s))


# --- RoPE ------------------------------------------------------------------------------

def _parse_closed(tok):
    if tok.startswith("cos("):
        return math.cos(float(tok[4:-1]))
    if tok.startswith("sin("):
        return math.sin(float(tok[4:-1]))
    return float(tok)


def test_rope_golden_cases():
    with open(os.path.join(GOLDEN, "rope_cases.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(lines) == 5
    for ln in lines:
        head, xs, exp = [p.split() for p in ln.split("|")]
        hd, theta, pos = int(head[0]), float(head[1]), float(head[2])
        x = np.array([float(v) for v in xs])[:, None]
        want = np.array([_parse_closed(v) for v in exp])
        assert x.shape[0] == hd
        got = oracle.rope_rotate(x, [pos], theta)[:, 0]
        np.testing.assert_allclose(got, want, atol=1e-12)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(5)
    hd, theta = 128, 1e6
    x = rng.standard_normal((hd, 7))
    pos = np.array([0, 1, 2, 17, 300, 4095, 8191])
    got = oracle.rope_rotate(x, pos, theta)
    half = hd // 2
    for t, p in enumerate(pos):
        for i in range(half):
            z = complex(x[i, t], x[i + half, t]) * np.exp(1j * p * theta ** (-2.0 * i / hd))
            assert abs(got[i, t] - z.real) < 1e-12
            assert abs(got[i + half, t] - z.imag) < 1e-12


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 5))
    np.testing.assert_array_equal(oracle.rope_rotate(x, np.zeros(5), 1e6), x)
    y = oracle.rope_rotate(x, np.array([1, 10, 100, 1000, 10000]), 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=0), np.linalg.norm(x, axis=0),
                               rtol=1e-13)


def test_rope_relative_position():
    # "LLM Speedrun: Architecture", RoPE: the dot product sees only the distance.
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal((32, 1)), rng.standard_normal((32, 1))
    a = (oracle.rope_rotate(q, [40], 1e4)[:, 0] @ oracle.rope_rotate(k, [13], 1e4)[:, 0])
    b = (oracle.rope_rotate(q, [127], 1e4)[:, 0] @ oracle.rope_rotate(k, [100], 1e4)[:, 0])
    assert abs(a - b) < 1e-12


def test_rope_frequencies_endpoints():
    f = oracle.rope_frequencies(128, 1e6)
    assert f.shape == (64,)
    assert f[0] == 1.0
    assert abs(f[63] - 1e6 ** (-126 / 128)) < 1e-18
    assert np.all(np.diff(f) < 0)


# --- softmax, RMSNorm, SiLU ------------------------------------------------------------

def test_softmax_closed_forms():
    np.testing.assert_allclose(oracle.softmax_rows(np.array([0.0, math.log(2.0)])),
                               [1 / 3, 2 / 3], rtol=1e-15)
    rng = np.random.default_rng(8)
    s = rng.standard_normal((4, 9)) * 30
    p = oracle.softmax_rows(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.softmax_rows(s + 123.0), p, rtol=1e-12)
    # a -1e9 entry contributes exactly zero
    assert oracle.softmax_rows(np.array([0.5, oracle.MASK_VALUE]))[1] == 0.0


def test_rms_norm_closed_forms():
    x = np.array([[3.0], [4.0]])
    np.testing.assert_allclose(oracle.rms_norm(x, np.ones(2), 0.0)[:, 0],
                               np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    c, eps = -0.25, 1e-6
    g = np.array([1.5, -2.0, 0.5])
    got = oracle.rms_norm(np.full((3, 1), c), g, eps)[:, 0]
    np.testing.assert_allclose(got, np.sign(c) * g * abs(c) / math.sqrt(c * c + eps),
                               rtol=1e-14)
    rng = np.random.default_rng(9)
    v = rng.standard_normal((50, 2))
    np.testing.assert_allclose(oracle.rms_norm(7.5 * v, np.ones(50), 0.0),
                               oracle.rms_norm(v, np.ones(50), 0.0), rtol=1e-13)


def test_silu_against_library_sigmoid():
    x = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(oracle.silu(x), x * expit(x), rtol=1e-13, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def test_zero_gate_gives_zero_mlp():
    m, w, s = tiny_model()
    m.w["model.layers.0.mlp.gate_proj.weight"] = np.zeros((s.intermediate, s.hidden))
    xn = np.random.default_rng(1).standard_normal((s.hidden, 3))
    np.testing.assert_array_equal(oracle.mlp_block(m, 0, xn), 0.0)


# --- attention -------------------------------------------------------------------------

def test_attention_single_key_returns_value():
    rng = np.random.default_rng(10)
    q, K, V = rng.standard_normal((16, 1)), rng.standard_normal((16, 1)), rng.standard_normal((16, 1))
    np.testing.assert_allclose(oracle.attend_one_head(q, K, V, [0], 16), V, rtol=1e-15)


def test_attention_zero_query_averages_open_values():
    rng = np.random.default_rng(11)
    K, V = rng.standard_normal((8, 6)), rng.standard_normal((8, 6))
    out = oracle.attend_one_head(np.zeros((8, 3)), K, V, [0, 2, 5], 8)
    for t, p in enumerate([0, 2, 5]):
        brute = sum(V[:, j] for j in range(p + 1)) / (p + 1)
        np.testing.assert_allclose(out[:, t], brute, rtol=1e-13)


def test_attention_ignores_future_keys():
    rng = np.random.default_rng(12)
    q, K, V = rng.standard_normal((8, 2)), rng.standard_normal((8, 6)), rng.standard_normal((8, 6))
    a = oracle.attend_one_head(q, K, V, [1, 3], 8)
    K2, V2 = K.copy(), V.copy()
    K2[:, 4:] += 100.0
    V2[:, 4:] -= 50.0
    np.testing.assert_allclose(oracle.attend_one_head(q, K2, V2, [1, 3], 8), a, rtol=1e-14)


def test_gqa_equals_mha_with_repeated_kv_heads():
    # "LLM Speedrun: Architecture", GQA: query heads share KV heads; the repeat of each
    # KV head over its consecutive group of query heads gives plain MHA.
    s = SHAPES["tiny"]
    w = make_weights(s)
    g = s.n_heads // s.n_kv_heads
    w_mha = dict(w)
    for li in range(s.n_layers):
        for nm in ("k_proj", "v_proj"):
            W = w[f"model.layers.{li}.self_attn.{nm}.weight"].reshape(s.n_kv_heads, s.head_dim, -1)
            b = w[f"model.layers.{li}.self_attn.{nm}.bias"].reshape(s.n_kv_heads, s.head_dim)
            w_mha[f"model.layers.{li}.self_attn.{nm}.weight"] = np.repeat(W, g, 0).reshape(-1, s.hidden)
            w_mha[f"model.layers.{li}.self_attn.{nm}.bias"] = np.repeat(b, g, 0).reshape(-1)
    cfg = OracleConfig.from_shape(s)
    cfg_mha = OracleConfig.from_shape(s)
    cfg_mha.n_kv_heads = s.n_heads
    ids = make_prompt(s, 6)
    t1, z1 = oracle.generate(OracleModel(cfg, w), ids, 4)
    t2, z2 = oracle.generate(OracleModel(cfg_mha, w_mha), ids, 4)
    assert t1 == t2
    for a, b in zip(z1, z2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_mha_config_runs_and_matches_bruteforce():
    m, w, s = tiny_model("mha_f32")
    ids = make_prompt(s, 3)
    _, z = oracle.step(m, list(ids), np.arange(3), oracle.KVCache(s.n_layers))
    np.testing.assert_allclose(z, brute_force_logits(w, s, list(ids)), rtol=0, atol=1e-10)


# --- causality and the KV cache ----------------------------------------------------------

def test_appending_tokens_never_changes_earlier_positions():
    m, w, s = tiny_model()
    ids = list(make_prompt(s, 8))
    full = oracle.forward_hidden(m, ids, np.arange(8), oracle.KVCache(s.n_layers))
    for n in (1, 3, 5):
        part = oracle.forward_hidden(m, ids[:n], np.arange(n), oracle.KVCache(s.n_layers))
        np.testing.assert_allclose(full[:, :n], part, rtol=0, atol=1e-13)


@pytest.mark.parametrize("shape", ["tiny", "small_f32"])
def test_cached_equals_uncached(shape):
    # "augur" (cached vs uncached generation) and the cache-free reference run of
    # "Building a Qwen2.5-1.5B Inference Engine From Scratch" §1.1 must agree.
    m, w, s = tiny_model(shape)
    ids = make_prompt(s, 8)
    t1, z1 = oracle.generate(m, ids, 8)
    t2, z2 = oracle.generate_uncached(m, ids, 8)
    assert t1 == t2
    for a, b in zip(z1, z2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_teacher_forcing_with_own_tokens_is_identity():
    m, w, s = tiny_model()
    ids = make_prompt(s, 8)
    t1, z1 = oracle.generate(m, ids, 6)
    t2, z2 = oracle.generate(m, ids, 6, feed=t1)
    assert t1 == t2
    for a, b in zip(z1, z2):
        np.testing.assert_array_equal(a, b)


def test_eos_is_appended_then_stops():
    m, w, s = tiny_model()
    ids = make_prompt(s, 8)
    t, _ = oracle.generate(m, ids, 8)
    t2, z2 = oracle.generate(m, ids, 8, eos=t[2])
    assert t2 == t[:t.index(t[2]) + 1]


def test_a_stop_set_stops_at_its_first_member():
    """generate_tokens' eos_ids: the first produced token found in the set ends the run
    (and is kept); ids that never come up do nothing; an empty set never stops."""
    m, w, s = tiny_model()
    ids = make_prompt(s, 8)
    t, _ = oracle.generate(m, ids, 10)
    absent = next(v for v in range(s.vocab) if v not in t)
    first = min(t.index(t[5]), t.index(t[3]))
    t2, _ = oracle.generate(m, ids, 10, eos_ids=[t[5], absent, t[3]])
    assert t2 == t[:first + 1]
    assert oracle.generate(m, ids, 10, eos_ids=[absent])[0] == t
    assert oracle.generate(m, ids, 10, eos_ids=[])[0] == t
    # the single eos and the set combine
    t3, _ = oracle.generate(m, ids, 10, eos=t[6], eos_ids=[absent])
    assert t3 == t[:t.index(t[6]) + 1]


# --- greedy choice ------------------------------------------------------------------------
# "augur", Features (greedy generation) and the argmax of the "LLM Speedrun: Architecture"
# model code: the largest logit wins; among equal maxima the lowest index (numpy's rule).

def test_greedy_takes_the_lowest_index_of_a_tie():
    assert oracle.greedy(np.array([1.0, 3.0, 3.0])) == 1
    assert oracle.greedy(np.array([3.0, 1.0, 3.0])) == 0
    assert oracle.greedy(np.array([-2.0, -1.0, -1.0, -5.0])) == 1


def test_greedy_ties_far_apart_and_at_the_end_of_a_full_vocabulary():
    V = 151936
    z = np.zeros(V)
    z[V - 2] = z[V - 1] = 1.0
    assert oracle.greedy(z) == V - 2
    z = np.full(V, -1.0)
    z[100000] = z[5] = 2.0
    assert oracle.greedy(z) == 5
    z = np.zeros(V)
    z[V - 1] = 1e-300  # a strictly larger last element still wins
    assert oracle.greedy(z) == V - 1


def test_greedy_agrees_with_a_scan_over_planted_ties():
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(1, 64))
        z = rng.integers(-3, 4, n).astype(np.float64)  # many equal values
        best = 0
        for i in range(1, n):  # the first strictly larger value moves the choice
            if z[i] > z[best]:
                best = i
        assert oracle.greedy(z) == best


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_greedy_rejects_non_finite_logits(bad):
    z = np.zeros(10)
    z[3] = bad
    with pytest.raises(FloatingPointError):
        oracle.greedy(z)


# --- optional weights: a separate LM head, no q/k/v bias ---------------------------------

def test_untied_head_copy_of_embedding_matches_tied():
    """A separate LM head equal to the embedding gives the tied model's logits exactly;
    a different head changes them, so the separate head is the one read."""
    s = SHAPES["untied_bf16"]
    w = make_weights(s)
    ids = make_prompt(s, 6)
    tied = OracleModel(OracleConfig.from_shape(s), w)
    tied.cfg.tied = True
    w_copy = dict(w)
    w_copy["lm_head.weight"] = w["model.embed_tokens.weight"].copy()
    untied_copy = OracleModel(OracleConfig.from_shape(s), w_copy)
    assert untied_copy.cfg.tied is False
    t1, z1 = oracle.generate(tied, ids, 4)
    t2, z2 = oracle.generate(untied_copy, ids, 4)
    assert t1 == t2
    for a, b in zip(z1, z2):
        np.testing.assert_array_equal(a, b)
    _, z3 = oracle.generate(OracleModel(OracleConfig.from_shape(s), w), ids, 1)
    assert np.max(np.abs(z3[0] - z1[0])) > 1e-3


def test_missing_qkv_bias_equals_zero_bias():
    s = SHAPES["untied_bf16"]
    w = make_weights(s)
    assert not any(k.endswith("_proj.bias") for k in w)
    w0 = dict(w)
    for i in range(s.n_layers):
        for name, n in (("q_proj", s.n_heads), ("k_proj", s.n_kv_heads), ("v_proj", s.n_kv_heads)):
            w0[f"model.layers.{i}.self_attn.{name}.bias"] = np.zeros(n * s.head_dim, dtype=np.float32)
    ids = make_prompt(s, 6)
    t1, z1 = oracle.generate(OracleModel(OracleConfig.from_shape(s), w), ids, 4)
    t2, z2 = oracle.generate(OracleModel(OracleConfig.from_shape(s), w0), ids, 4)
    assert t1 == t2
    for a, b in zip(z1, z2):
        np.testing.assert_array_equal(a, b)


# --- closed-form reduction: zero blocks --------------------------------------------------

def test_zero_blocks_reduce_to_normed_embedding_logits():
    s = SHAPES["tiny"]
    w = make_weights(s)
    for k in list(w):
        if k.startswith("model.layers.") and not k.endswith("layernorm.weight"):
            w[k] = np.zeros_like(w[k])
    m = OracleModel(OracleConfig.from_shape(s), w)
    ids = list(make_prompt(s, 5))
    _, z = oracle.step(m, ids, np.arange(5), oracle.KVCache(s.n_layers))
    E = w["model.embed_tokens.weight"].astype(np.float64)
    wf = w["model.norm.weight"].astype(np.float64)
    e = E[ids[-1]]
    r = math.sqrt(sum(float(v) ** 2 for v in e) / s.hidden + s.rms_eps)
    for tok in range(s.vocab):
        want = sum(float(E[tok, i]) * float(wf[i]) * float(e[i]) / r for i in range(s.hidden))
        assert abs(z[tok] - want) < 1e-12


# --- brute force: independent scalar loops on the tiny shape ----------------------------

def brute_force_logits(w, s, ids):
    """Scalar-loop restatement, row-major, one token at a time over explicit lists."""
    H, hd, nq, nkv = s.hidden, s.head_dim, s.n_heads, s.n_kv_heads
    half = hd // 2
    W = {k: v.astype(np.float64).tolist() for k, v in w.items()}

    def matvec(M, x):
        return [sum(r[i] * x[i] for i in range(len(x))) for r in M]

    def norm(x, g):
        ms = sum(v * v for v in x) / len(x)
        inv = 1.0 / math.sqrt(ms + s.rms_eps)
        return [x[i] * inv * g[i] for i in range(len(x))]

    def rot(vec, pos):
        out = list(vec)
        for i in range(half):
            ang = pos * (s.rope_theta ** (-(2.0 * i) / hd))
            a, b = vec[i], vec[i + half]
            out[i] = a * math.cos(ang) - b * math.sin(ang)
            out[i + half] = b * math.cos(ang) + a * math.sin(ang)
        return out

    xs = [list(W["model.embed_tokens.weight"][t]) for t in ids]
    for li in range(s.n_layers):
        p = f"model.layers.{li}."
        Ks = [[] for _ in range(nkv)]
        Vs = [[] for _ in range(nkv)]
        Qs = []
        for pos, x in enumerate(xs):
            n = norm(x, W[p + "input_layernorm.weight"])
            q = [a + b for a, b in zip(matvec(W[p + "self_attn.q_proj.weight"], n), W[p + "self_attn.q_proj.bias"])]
            k = [a + b for a, b in zip(matvec(W[p + "self_attn.k_proj.weight"], n), W[p + "self_attn.k_proj.bias"])]
            v = [a + b for a, b in zip(matvec(W[p + "self_attn.v_proj.weight"], n), W[p + "self_attn.v_proj.bias"])]
            Qs.append([rot(q[h * hd:(h + 1) * hd], pos) for h in range(nq)])
            for g in range(nkv):
                Ks[g].append(rot(k[g * hd:(g + 1) * hd], pos))
                Vs[g].append(v[g * hd:(g + 1) * hd])
        new_xs = []
        for pos, x in enumerate(xs):
            o = []
            for h in range(nq):
                g = h // (nq // nkv)
                sc = [sum(Qs[pos][h][d] * Ks[g][j][d] for d in range(hd)) / math.sqrt(H / nq)
                      for j in range(pos + 1)]
                mx = max(sc)
                ex = [math.exp(v - mx) for v in sc]
                tot = sum(ex)
                o += [sum(ex[j] / tot * Vs[g][j][d] for j in range(pos + 1)) for d in range(hd)]
            h1 = [a + b for a, b in zip(x, matvec(W[p + "self_attn.o_proj.weight"], o))]
            n2 = norm(h1, W[p + "post_attention_layernorm.weight"])
            gt = matvec(W[p + "mlp.gate_proj.weight"], n2)
            up = matvec(W[p + "mlp.up_proj.weight"], n2)
            act = [u * (gv / (1.0 + math.exp(-gv))) for gv, u in zip(gt, up)]
            new_xs.append([a + b for a, b in zip(h1, matvec(W[p + "mlp.down_proj.weight"], act))])
        xs = new_xs
    hf = norm(xs[-1], W["model.norm.weight"])
    return np.array(matvec(W["model.embed_tokens.weight"], hf))


@pytest.mark.parametrize("shape,n", [("tiny", 4), ("small_f32", 3)])
def test_oracle_matches_scalar_bruteforce(shape, n):
    m, w, s = tiny_model(shape)
    ids = list(make_prompt(s, n))
    _, z = oracle.step(m, ids, np.arange(n), oracle.KVCache(s.n_layers))
    np.testing.assert_allclose(z, brute_force_logits(w, s, ids), rtol=0, atol=1e-10)


# --- input generator vs a library routine --------------------------------------------------

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    a = (rng.standard_normal(100000) * 0.02).astype(np.float32)
    # exact ties: low 16 bits 0x8000 with even and odd upper halves
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3C238000], dtype=np.uint32).view(np.float32)
    a = np.concatenate([a, ties])
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(round_to_bf16(a), want)


def test_weights_are_deterministic_and_layer_subsets_agree():
    s = SHAPES["small_bf16"]
    a = make_weights(s)
    b = make_weights(s, layers=[1])
    for k, v in b.items():
        np.testing.assert_array_equal(a[k], v)
    assert "model.layers.0.mlp.up_proj.weight" not in b
    g = a["model.layers.0.input_layernorm.weight"]
    assert abs(g.mean() - 1.0) < 0.01 and 0.01 < g.std() < 0.03
    wq = a["model.layers.0.self_attn.q_proj.weight"]
    assert abs(wq.std() - 0.02) < 0.001
    np.testing.assert_array_equal(round_to_bf16(wq), wq)


# --- float32 mode (the timed CPU baseline) ----------------------------------------------

@pytest.mark.parametrize("shape", ["tiny", "small_f32"])
def test_float32_mode_stays_float32_and_follows_float64(shape):
    # The float32 mode runs the float64 oracle's steps in the precision of the numpy model
    # code on "LLM Speedrun: Architecture" (every array float32). It must keep its arrays
    # float32 (else it would not time float32 BLAS) and agree with the pinned float64 oracle
    # to float32 rounding: the same greedy tokens under teacher forcing, logits within 1e-4 of
    # their spread.
    m64, w, s = tiny_model(shape)
    m32 = OracleModel(OracleConfig.from_shape(s), w, dtype=np.float32)
    assert all(v.dtype == np.float32 for v in m32.w.values())
    prompt = make_prompt(s, 12)
    t64, z64 = oracle.generate(m64, prompt, 6)
    t32, z32 = oracle.generate(m32, prompt, 6, feed=t64[:-1])
    assert all(z.dtype == np.float32 for z in z32)
    assert all(z.dtype == np.float64 for z in z64)
    for a, b in zip(z64, z32):
        assert np.max(np.abs(a - b)) <= 1e-4 * np.std(a)
    assert t32 == t64
