"""GB300-native MoE dispatch / combine (DeepEP-style expert-parallel exchange).

The compute path is ``libep.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/ep.h``); this package is its thin Python binding.
"""
