"""GB300-native batch-one Qwen3 decoder: the C-ABI library libqw.so and its binding.

The decoder forward (prefill and greedy decode) runs in hand-written sm_103a kernels
behind include/qw.h; ``qw`` is the ctypes binding, ``build`` compiles the library.
"""
from . import qw  # noqa: F401
from .qw import Model, QwError, weights_to_device  # noqa: F401
