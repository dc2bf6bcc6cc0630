"""GB300-native forward hot path of a nano-vllm-style Qwen3 engine.

The compute runs in libqw.so (hand-written CUDA for sm_103a, C ABI in
include/qw.h); this package binds it (``_lib``) and sequences it
(``model``).  PyTorch provides device memory and streams only.
"""
from . import _lib as lib  # noqa: F401
from ._lib import QwError  # noqa: F401

__all__ = ["lib", "QwError", "model", "build"]
