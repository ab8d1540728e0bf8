"""GB300-native forward pass of an FP4-expert MoE layer.

The compute path lives in the CUDA library built from ``csrc/`` (loaded by
``fp4_expert_grouped_gb300.capi``); this package only marshals arguments to it.
Importing the package itself loads nothing, so that the synthetic-input module
(``inputs``) can be used on machines without the library.
"""
__all__ = ["capi", "inputs"]
