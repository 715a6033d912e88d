"""ctypes binding of libqw's C ABI (argument marshalling only).

Every step of the forward pass runs in libqw's CUDA kernels; this module only converts
Python values to the C structs, uploads weights into one device buffer (PyTorch holds the
memory) and forwards calls. There is no fallback: if the library is missing, loading
fails with an error.
"""
import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqw.so")

QW_OK = 0
STATUS = {
    0: "QW_OK", 1: "QW_ERR_INVALID_ARG", 2: "QW_ERR_UNSUPPORTED", 3: "QW_ERR_CAPACITY",
    4: "QW_ERR_TOKEN_RANGE", 5: "QW_ERR_CUDA", 6: "QW_ERR_TIMEOUT",
    7: "QW_ERR_FAULT_INJECTED", 8: "QW_ERR_NUMERIC",
}
F32, BF16, F16 = 0, 1, 2


class QwError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class QwConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "intermediate", "vocab")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("tied_embeddings", ctypes.c_int32), ("qkv_bias", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("max_seqs", ctypes.c_int32), ("kv_capacity", ctypes.c_int32)]


_LAYER_FIELDS = ("in_norm", "wq", "bq", "wk", "bk", "wv", "bv", "wo", "post_norm", "w_gate",
                 "w_up", "w_down")


class QwLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYER_FIELDS]


class QwWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("layers", ctypes.POINTER(QwLayerWeights))]


_lib = None


def lib():
    """Load libqw.so (built by ``__graft_entry__.build()``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, VP, SZ = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    pi = P(I32)
    sig = {
        "qw_create": ([P(QwConfig), P(QwWeights), VP, P(VP)], I32),
        "qw_destroy": ([VP], None),
        "qw_prefill": ([VP, I32, pi, I32, pi], I32),
        "qw_prefill_device": ([VP, I32, VP, I32], I32),
        "qw_decode_step": ([VP, pi, pi], I32),
        "qw_decode_steps": ([VP, I32], I32),
        "qw_generate": ([VP, pi, I32, I32, I32, pi, pi], I32),
        "qw_generate_stops": ([VP, pi, I32, I32, pi, I32, pi, pi], I32),
        "qw_sync": ([VP], I32),
        "qw_logits": ([VP], VP),
        "qw_read_logits": ([VP, I32, P(ctypes.c_float)], I32),
        "qw_tokens_device": ([VP], VP),
        "qw_decode_kernels_per_step": ([VP], I32),
        "qw_position": ([VP, I32, pi], I32),
        "qw_reset": ([VP, I32], I32),
        "qw_last_error": ([], ctypes.c_char_p),
        "qw_set_trace": ([VP, I32, P(VP), P(VP)], I32),
        "qw_set_timeline": ([VP, I32], I32),
        "qw_read_timeline": ([VP, P(ctypes.c_uint64), I32, pi], I32),
        "qw_op_decode_attention_noalloc": ([I32, I32, I32, I32, I32, I32, VP, VP, VP, VP, VP], I32),
        "qw_op_decode_attention_noalloc_limit": ([], SZ),
        "qw_op_gemm_f16": ([I32, I32, I32, VP, VP, VP, VP, I32, VP, VP], I32),
        "qw_op_gemm_swiglu_f16": ([I32, I32, I32, VP, VP, VP, VP, VP, VP], I32),
        "qw_op_decode_attention_workspace": ([I32, I32, I32, I32], SZ),
        "qw_op_decode_attention": ([I32, I32, I32, I32, I32, I32, VP, VP, VP, VP, VP, SZ, VP], I32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def exported_symbols():
    return ["qw_create", "qw_destroy", "qw_prefill", "qw_prefill_device", "qw_decode_step",
            "qw_decode_steps", "qw_generate", "qw_generate_stops", "qw_sync", "qw_logits", "qw_read_logits",
            "qw_tokens_device", "qw_decode_kernels_per_step", "qw_position", "qw_reset",
            "qw_last_error", "qw_set_trace",
            "qw_set_timeline", "qw_read_timeline",
            "qw_op_decode_attention_workspace", "qw_op_decode_attention",
            "qw_op_decode_attention_noalloc", "qw_op_decode_attention_noalloc_limit", "qw_op_gemm_f16",
            "qw_op_gemm_swiglu_f16"]


def check(status):
    if status != QW_OK:
        raise QwError(status, lib().qw_last_error().decode())


def _iptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class DeviceWeights:
    """All tensors of one model in a single device buffer, each 256-byte aligned.

    ``arrays`` maps parameter names to float32 numpy arrays; for bf16 models every value
    must already be exactly representable in bf16 (the synthetic generator rounds)."""

    def __init__(self, arrays: dict, dtype: int, device="cuda"):
        import torch
        self.dtype = dtype
        esize = 2 if dtype == BF16 else 4
        offs, total = {}, 0
        for k, a in arrays.items():
            offs[k] = total
            total += (a.size * esize + 255) // 256 * 256
        self.buf = torch.empty(total, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        self.ptr = {}
        for k, a in arrays.items():
            a = np.ascontiguousarray(a, dtype=np.float32)
            if dtype == BF16:
                u = (a.view(np.uint32) >> 16).astype(np.uint16)
                src = torch.from_numpy(u.view(np.int16).reshape(-1)).view(torch.uint8)
            else:
                src = torch.from_numpy(a.reshape(-1)).view(torch.uint8)
            o = offs[k]
            self.buf[o:o + src.numel()].copy_(src)
            self.ptr[k] = base + o
        self.nbytes = total


class Model:
    """One libqw model over borrowed device weights."""

    def __init__(self, shape, dev_weights: DeviceWeights, kv_capacity, max_seqs=1, stream=None):
        L = lib()
        self.shape = shape
        self.weights = dev_weights  # keep the device buffer alive
        dt = BF16 if shape.dtype == "bf16" else F32
        cfg = QwConfig(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads,
                       shape.head_dim, shape.intermediate, shape.vocab, shape.rms_eps,
                       shape.rope_theta, int(shape.tied), int(shape.qkv_bias), dt, max_seqs,
                       kv_capacity)
        p = dev_weights.ptr
        layers = (QwLayerWeights * shape.n_layers)()
        for i in range(shape.n_layers):
            pre = f"model.layers.{i}."
            names = {
                "in_norm": "input_layernorm.weight", "wq": "self_attn.q_proj.weight",
                "bq": "self_attn.q_proj.bias", "wk": "self_attn.k_proj.weight",
                "bk": "self_attn.k_proj.bias", "wv": "self_attn.v_proj.weight",
                "bv": "self_attn.v_proj.bias", "wo": "self_attn.o_proj.weight",
                "post_norm": "post_attention_layernorm.weight", "w_gate": "mlp.gate_proj.weight",
                "w_up": "mlp.up_proj.weight", "w_down": "mlp.down_proj.weight"}
            for f, n in names.items():
                setattr(layers[i], f, p.get(pre + n))
        w = QwWeights(p["model.embed_tokens.weight"], p["model.norm.weight"],
                      p.get("lm_head.weight"), layers)
        self._layers = layers
        h = ctypes.c_void_p()
        check(L.qw_create(ctypes.byref(cfg), ctypes.byref(w), stream, ctypes.byref(h)))
        self.h = h
        self.max_seqs = max_seqs
        self.kv_capacity = kv_capacity

    def close(self):
        if self.h:
            lib().qw_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, ids, seq=0):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        out = np.zeros(1, dtype=np.int32)
        check(lib().qw_prefill(self.h, seq, _iptr(ids), len(ids), _iptr(out)))
        return int(out[0])

    def prefill_device(self, ids_dev_ptr, n, seq=0):
        check(lib().qw_prefill_device(self.h, seq, ids_dev_ptr, n))

    def decode_step(self, feed=None):
        """One decode step of every active sequence; returns the new tokens [max_seqs]."""
        out = np.zeros(self.max_seqs, dtype=np.int32)
        f = None
        if feed is not None:
            f = np.ascontiguousarray(np.broadcast_to(feed, (self.max_seqs,)), dtype=np.int32)
        check(lib().qw_decode_step(self.h, _iptr(f) if f is not None else None, _iptr(out)))
        return out

    def decode_steps(self, n):
        check(lib().qw_decode_steps(self.h, n))

    def generate(self, ids, max_new, eos=-1, eos_ids=None):
        """Greedy generation of sequence 0; stops after a token equal to eos (eos >= 0) or
        to any id of eos_ids (qw_generate_stops), which is kept."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        out = np.zeros(max_new, dtype=np.int32)
        n_out = np.zeros(1, dtype=np.int32)
        if eos_ids is None:
            check(lib().qw_generate(self.h, _iptr(ids), len(ids), max_new, eos, _iptr(out), _iptr(n_out)))
        else:
            stops = np.ascontiguousarray(list(eos_ids) + ([eos] if eos >= 0 else []), dtype=np.int32)
            check(lib().qw_generate_stops(self.h, _iptr(ids), len(ids), max_new, _iptr(stops), len(stops),
                                          _iptr(out), _iptr(n_out)))
        return out[:int(n_out[0])].tolist()

    def sync(self):
        check(lib().qw_sync(self.h))

    def logits(self, seq=0):
        z = np.empty(self.shape.vocab, dtype=np.float32)
        check(lib().qw_read_logits(self.h, seq, z.ctypes.data_as(ctypes.POINTER(ctypes.c_float))))
        return z

    def logits_ptr(self):
        return lib().qw_logits(self.h)

    def tokens_ptr(self):
        return lib().qw_tokens_device(self.h)

    def decode_kernels_per_step(self):
        """1 when a single-sequence decode step runs as one persistent kernel."""
        return int(lib().qw_decode_kernels_per_step(self.h))

    def position(self, seq=0):
        p = np.zeros(1, dtype=np.int32)
        check(lib().qw_position(self.h, seq, _iptr(p)))
        return int(p[0])

    def set_trace(self, kind, begin_events=None, end_events=None):
        """Record CUDA events (torch.cuda.Event, timing enabled) around kernel ``kind`` of
        every layer in later decode steps; None removes the hook."""
        if begin_events is None:
            check(lib().qw_set_trace(self.h, kind, None, None))
            return
        n = len(begin_events)
        b = (ctypes.c_void_p * n)(*[e.cuda_event for e in begin_events])
        e = (ctypes.c_void_p * n)(*[x.cuda_event for x in end_events])
        self._trace_keep = (b, e, begin_events, end_events)
        check(lib().qw_set_trace(self.h, kind, b, e))

    def set_timeline(self, enable=True):
        check(lib().qw_set_timeline(self.h, int(enable)))

    def read_timeline(self):
        """[(start_ns, wait_released_ns, end_ns)] per kernel of the last decode step."""
        # a batched step launches the most kernels; the persistent step kernel writes three
        # records per phase and per-CTA barrier arrivals
        n_max = max(3 + 10 * self.shape.n_layers, 3 * (5 * self.shape.n_layers + 1) + 2048)
        buf = (ctypes.c_uint64 * (3 * n_max))()
        n = np.zeros(1, dtype=np.int32)
        check(lib().qw_read_timeline(self.h, buf, n_max, _iptr(n)))
        a = np.frombuffer(buf, dtype=np.uint64)[:3 * int(n[0])].reshape(-1, 3)
        return a

    def reset(self, seq=0):
        check(lib().qw_reset(self.h, seq))


def decode_attention(dtype, n_heads, n_kv_heads, head_dim, ctx, kv_stride, q_ptr, k_ptr, v_ptr,
                     out_ptr, ws_ptr, ws_bytes, stream=None):
    check(lib().qw_op_decode_attention(dtype, n_heads, n_kv_heads, head_dim, ctx, kv_stride,
                                       q_ptr, k_ptr, v_ptr, out_ptr, ws_ptr, ws_bytes, stream))


def decode_attention_noalloc(kv_dtype, n_heads, n_kv_heads, head_dim, ctx, kv_stride, q_ptr, k_ptr,
                             v_ptr, out_ptr, stream=None):
    """Decode attention whose scratch is the library's fixed array (no allocation)."""
    check(lib().qw_op_decode_attention_noalloc(kv_dtype, n_heads, n_kv_heads, head_dim, ctx,
                                               kv_stride, q_ptr, k_ptr, v_ptr, out_ptr, stream))


def decode_attention_workspace(n_heads, n_kv_heads, head_dim, max_ctx):
    return int(lib().qw_op_decode_attention_workspace(n_heads, n_kv_heads, head_dim, max_ctx))


def gemm_f16(M, N, K, a_ptr, b_ptr, bias_ptr, c_ptr, accumulate, err_ptr, stream=None):
    check(lib().qw_op_gemm_f16(M, N, K, a_ptr, b_ptr, bias_ptr, c_ptr, int(accumulate), err_ptr, stream))


def gemm_swiglu_f16(M, N, K, a_ptr, wg_ptr, wu_ptr, act_ptr, err_ptr, stream=None):
    check(lib().qw_op_gemm_swiglu_f16(M, N, K, a_ptr, wg_ptr, wu_ptr, act_ptr, err_ptr, stream))
