"""GB300-native MoE dispatch / combine (DeepEP-style expert-parallel exchange).

The compute path is ``libep.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/ep.h``); ``ep`` is its thin binding (same names as the C
entry points) and ``Buffer`` the DeepEP-style object API on top.  Importing
the package does not load the library; the first call does, and fails loudly
if it has not been built.
"""


def __getattr__(name):
    if name in ("Buffer", "Handle"):
        from . import buffer
        return getattr(buffer, name)
    raise AttributeError(name)
