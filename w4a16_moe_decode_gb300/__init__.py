"""GB300-native (sm_103a) small-batch decode step of a Flint-style MoE FFN
layer with weight-only NVFP4 (W4A16) weights and BF16 activations.

The computation lives in libflint_moe.so (C ABI: include/flint_moe.h);
``binding`` exposes its entry points under the same names.
"""
from . import binding  # noqa: F401
from .build import LIB, build  # noqa: F401
