"""GB300-native (sm_103a) DFlash + DDTree speculative step.

The compute lives in ``libdflash.so`` (CUDA kernels behind the C ABI in
``include/dflash.h``); ``_lib`` is its ctypes binding and ``engine`` drives a step.
"""
from . import _lib  # noqa: F401
from ._lib import StatusError, Workspace, load  # noqa: F401
