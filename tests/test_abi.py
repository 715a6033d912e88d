"""The C ABI library loads, exports every symbol include/qw.h declares, and rejects bad
arguments before touching a GPU (these tests need none)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from qwen2_decoder_forward_decode_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return binding.lib()


def header_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(qw_\w+)\s*\(", text))
    return names


def test_every_declared_function_is_exported(L):
    declared = header_functions()
    assert {"qw_create", "qw_prefill", "qw_decode_step", "qw_generate"} <= declared
    for name in sorted(declared):
        assert hasattr(L, name), f"{name} declared in include/ but not exported"
    assert declared == set(binding.exported_symbols())


def _cfg(**over):
    c = dict(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, intermediate=128,
             vocab=256, rms_eps=1e-6, rope_theta=1e6, tied_embeddings=1, qkv_bias=1, dtype=0,
             max_seqs=1, kv_capacity=16)
    c.update(over)
    return binding.QwConfig(**c)


def _weights(n_layers=2, align=256, null=None):
    fake = 0x10000000
    layers = (binding.QwLayerWeights * n_layers)()
    for i in range(n_layers):
        for j, f in enumerate(binding._LAYER_FIELDS):
            setattr(layers[i], f, fake + align * (i * 16 + j + 1))
    if null:
        setattr(layers[0], null, None)
    return binding.QwWeights(fake, fake + align, None, layers), layers


def _create(L, cfg, w):
    h = ctypes.c_void_p()
    st = L.qw_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h))
    return st, L.qw_last_error().decode()


@pytest.mark.parametrize("over,status", [
    (dict(hidden=0), 1),
    (dict(head_dim=15), 1),
    (dict(n_kv_heads=3), 1),
    (dict(hidden=96), 2),            # head_dim != hidden / n_heads
    (dict(head_dim=8, hidden=32), 2),  # head_dim without a kernel
    (dict(dtype=7), 1),
    (dict(max_seqs=17), 2),
    (dict(kv_capacity=0), 1),
    (dict(n_heads=36, n_kv_heads=4, hidden=576), 2),  # 9 query heads per KV head
])
def test_bad_config_rejected(L, over, status):
    w, _keep = _weights()
    st, msg = _create(L, _cfg(**over), w)
    assert st == status, msg
    assert msg


def test_null_and_misaligned_weights_rejected(L):
    w, _keep = _weights(null="wo")
    st, msg = _create(L, _cfg(), w)
    assert st == 1 and "null" in msg
    w, _keep = _weights(align=8)
    st, msg = _create(L, _cfg(), w)
    assert st == 1 and "aligned" in msg
    w, _keep = _weights()
    st, msg = _create(L, _cfg(tied_embeddings=0), w)
    assert st == 1 and "lm_head" in msg


def test_null_arguments(L):
    assert L.qw_prefill(None, 0, None, 1, None) == 1
    assert L.qw_decode_step(None, None, None) == 1
    assert L.qw_generate(None, None, 1, 1, -1, None, None) == 1
    assert L.qw_sync(None) == 1
    assert L.qw_logits(None) is None
    assert L.qw_op_decode_attention_workspace(12, 2, 128, 0) == 0
    assert L.qw_op_decode_attention(1, 12, 2, 128, 1, 1, None, None, None, None, None, 0, None) == 1


def test_attention_workspace_size_grows_with_context(L):
    a = L.qw_op_decode_attention_workspace(12, 2, 128, 64)
    b = L.qw_op_decode_attention_workspace(12, 2, 128, 8192)
    assert 0 < a < b


@pytest.mark.skipif(os.environ.get("CUDA_VISIBLE_DEVICES") is None and os.path.exists("/dev/nvidia0"),
                    reason="only meaningful on a machine without a GPU")
def test_valid_config_without_gpu_fails_loudly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    w, _keep = _weights()
    st, msg = _create(L, _cfg(), w)
    assert st == 5, msg  # QW_ERR_CUDA: no silent CPU path


def test_fault_injection_at_create_then_the_library_still_works(L, monkeypatch):
    """QW_FAULT=alloc makes qw_create fail with QW_ERR_FAULT_INJECTED after validation and
    before any device work; without it the same call proceeds normally again."""
    w, _keep = _weights()
    monkeypatch.setenv("QW_FAULT", "alloc")
    st, msg = _create(L, _cfg(), w)
    assert st == 7 and "QW_FAULT" in msg
    st, msg = _create(L, _cfg(hidden=0), w)  # validation still comes first
    assert st == 1
    monkeypatch.delenv("QW_FAULT")
    st, msg = _create(L, _cfg(), w)
    assert st != 7
    if st == 0:
        pytest.skip("a GPU is present: the model was created")
    assert st == 5  # no GPU here: QW_ERR_CUDA


def test_last_error_is_cleared_by_the_next_call(L):
    assert L.qw_reset(None, 0) == 1
    assert L.qw_last_error().decode()
    assert L.qw_op_decode_attention_workspace(12, 2, 128, 64) > 0  # (sets no error)
    assert L.qw_position(None, 0, None) == 1
    msg = L.qw_last_error().decode()
    assert msg and "null" in msg
