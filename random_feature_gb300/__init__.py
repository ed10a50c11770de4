"""FAVOR+ forward attention (Performers) for one GB300: a C-ABI CUDA library
(libfavor.so, kernels for sm_103a) and its ctypes binding."""
from .favor import *  # noqa: F401,F403
from .favor import __all__  # noqa: F401
