"""LatentMoE layer forward pass on GB300 (sm_103a): Python binding over the C-ABI library.

The binding (``LatentMoE``) is imported lazily so that ``configs`` and ``inputs`` can be used
without the CUDA library present.
"""


def __getattr__(name):
    if name in ("LatentMoE", "LatentMoEError"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
