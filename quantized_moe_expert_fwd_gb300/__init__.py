"""GB300-native routed MoE FFN forward (int4 g32 SwiGLU experts, top-K router,
sigmoid-gated shared expert).

The computation lives in libstrata_moe.so (hand-written sm_103a CUDA behind
the C ABI of include/strata_moe.h); this package builds it (build.py), binds
it (strata_moe.py) and packs canonical weights into its layout (pack.py).
"""
from . import build  # noqa: F401
from .strata_moe import *  # noqa: F401,F403
from .strata_moe import DeviceLayer, StrataError, load, make_workspace  # noqa: F401
