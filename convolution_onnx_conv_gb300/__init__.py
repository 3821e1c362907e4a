"""Fused ONNX Conv (+ folded inference BatchNorm, bias, ReLU/ReLU6/Clip) for GB300 (sm_103a).

The compute lives in ``libconvfused.so`` (hand-written CUDA for sm_103a, C ABI declared in
``include/conv_fused.h``); this package is its ctypes binding plus the shape tables and the
seeded synthetic inputs of the workloads.  Importing it does not load the library; the first
call does, and fails loudly if the library is not built.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import (ConvDesc, ConvFusedError, FusedConv, ConvChain, load_library, make_desc,  # noqa: F401
                       library_path, EXPORTED, VARIANT_NAMES)
