"""GB300-native small-M routed-MoE decode/verify layer.

The layer (router GEMV -> softmax top-k -> SwiGLU experts -> weighted
combine) runs in hand-written sm_103a CUDA kernels behind the C ABI in
``include/moe.h``; ``MoELayer`` is its Python face.  ``LmHead`` is the bf16
vocabulary projection of the same decode step (``include/lm_head.h``).  Importing the package
loads nothing; the CUDA library is loaded (and must exist) on first use.
"""

__all__ = ["MoELayer", "LmHead", "tp_slice", "combine_partials"]


def __getattr__(name):
    if name in __all__:
        from . import layer
        return getattr(layer, name)
    raise AttributeError(name)
