"""GB300 (sm_103a) Qwen2 decoder forward pass: KV-cached greedy decode and prefill.

The compute lives in ``libqw.so`` (CUDA kernels behind a C ABI, ``include/qw.h``);
``binding`` marshals Python values into those calls. Build with ``build.build()``.
"""
from . import binding  # noqa: F401
from .binding import Model, DeviceWeights, QwError, lib  # noqa: F401

__all__ = ["binding", "Model", "DeviceWeights", "QwError", "lib"]
