"""GB300-native forward pass of a top-k gated Mixture-of-Experts FFN layer.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``include/moe.h``); :mod:`.lib` is its Python binding. Importing
this package does not load the library; :func:`lib.load` does, and fails
loudly if it has not been built.
"""
from .configs import CONFIGS, LayerConfig  # noqa: F401

__all__ = ["CONFIGS", "LayerConfig"]
