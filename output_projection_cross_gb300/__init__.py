"""GB300-native fused LM-head loss: Python binding of liblossk.so.

The compute path is the C ABI declared in include/lossk.h and implemented by
hand-written sm_103a CUDA kernels under csrc/.  This package only marshals
torch tensors into those calls (see lossk.py); importing it fails loudly when
the library has not been built.
"""
from .lossk import *  # noqa: F401,F403
from .lossk import LosskError, lib, workspace  # noqa: F401
