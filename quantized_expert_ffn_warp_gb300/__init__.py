"""GB300 (sm_103a) quantised MoE layer forward for decode and small-batch serving.

The compute path is the C-ABI library libmoe_layer.so (include/moe_layer.h);
``moe`` is its thin Python binding and ``synth`` draws seeded synthetic layers.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "moe", "build"]
