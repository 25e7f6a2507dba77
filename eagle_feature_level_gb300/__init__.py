"""GB300-native EAGLE / EAGLE-2 draft-and-verify round.

The compute path is libeagle.so (hand-written CUDA for sm_103a, C ABI in
include/eagle.h); this package binds it (`_binding`, same names as the C
functions) and sequences its calls over torch-allocated buffers
(`runtime`).  There is no CPU fallback: importing the binding of an unbuilt
library raises.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import EagleError, lib  # noqa: F401
from .build import build  # noqa: F401
