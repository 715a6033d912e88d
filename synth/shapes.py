"""Model shapes and run recipes for the synthetic Qwen2-style decoders.

The Qwen2.5 shapes follow the model configurations named on the pages
("Building a Qwen2.5-1.5B Inference Engine From Scratch", §1.1: 28 layers, 12 query
heads, 2 key-value heads; "augur", Features: hidden size, head counts, MLP size,
RMSNorm epsilon, RoPE theta, vocabulary size). The small shapes exist so parity tests
span several tiles with ragged tails while the oracle still finishes in seconds.
"""
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Shape:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    dtype: str  # "f32" or "bf16": storage type of weights and KV cache
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    tied: bool = True
    qkv_bias: bool = True

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads


@dataclass(frozen=True)
class Workload:
    name: str
    shape: str
    prompt_len: int          # single-sequence prompt length (0 for batched)
    new_tokens: int          # tokens produced in total, the prefill's one included
    kv_capacity: int
    n_seqs: int = 1
    batch_len_range: tuple = field(default=(0, 0))  # inclusive [lo, hi] for batched


SHAPES = {
    # 2 layers, hidden 64, 4/2 heads, head_dim 16, MLP 128, vocab 256, fp32
    "tiny": Shape("tiny", 2, 64, 4, 2, 16, 128, 256, "f32"),
    # Qwen2.5-0.5B shape, bf16
    "0p5b": Shape("0p5b", 24, 896, 14, 2, 64, 4864, 151936, "bf16"),
    # Qwen2.5-1.5B shape, bf16
    "1p5b": Shape("1p5b", 28, 1536, 12, 2, 128, 8960, 151936, "bf16"),
    # Qwen2.5-Coder-7B shape, bf16 (28 query / 4 KV heads: 7 per group; MLP 18944), and its
    # first two layers with the full widths and vocabulary for parity runs
    "7b": Shape("7b", 28, 3584, 28, 4, 128, 18944, 152064, "bf16"),
    "7b_2l": Shape("7b_2l", 2, 3584, 28, 4, 128, 18944, 152064, "bf16"),
    # small shapes with ragged tails for fast parity tests
    "small_bf16": Shape("small_bf16", 2, 384, 6, 2, 64, 1000, 3001, "bf16"),
    "small_f32": Shape("small_f32", 3, 96, 3, 1, 32, 200, 1000, "f32"),
    "mha_f32": Shape("mha_f32", 2, 64, 4, 4, 16, 96, 300, "f32"),
    "hd128_bf16": Shape("hd128_bf16", 2, 768, 6, 2, 128, 2304, 5000, "bf16"),
    # even query heads per KV head (4 and 2), head sizes 64 and 128
    "gqa4_bf16": Shape("gqa4_bf16", 2, 512, 8, 2, 64, 1024, 3001, "bf16"),
    "gqa2_hd128_bf16": Shape("gqa2_hd128_bf16", 2, 512, 4, 2, 128, 1408, 3001, "bf16"),
    # the optional weights switched the other way: a separate LM head, no q/k/v bias
    "untied_bf16": Shape("untied_bf16", 2, 256, 4, 2, 64, 704, 2051, "bf16", tied=False, qkv_bias=False),
}


WORKLOADS = {
    "tiny": Workload("tiny", "tiny", prompt_len=8, new_tokens=8, kv_capacity=16),
    "0p5b": Workload("0p5b", "0p5b", prompt_len=32, new_tokens=32, kv_capacity=64),
    "1p5b": Workload("1p5b", "1p5b", prompt_len=128, new_tokens=100, kv_capacity=2048),
    "1p5b_long": Workload("1p5b_long", "1p5b", prompt_len=4096, new_tokens=256,
                          kv_capacity=8192),
    "1p5b_batch": Workload("1p5b_batch", "1p5b", prompt_len=0, new_tokens=128,
                           kv_capacity=2304, n_seqs=16, batch_len_range=(256, 2048)),
}
