"""Windowed-KV-cache GroupQueryAttention for GB300 (sm_103a).

The computation lives in ``libgqaw.so`` (CUDA kernels behind the C ABI of
include/gqaw.h); :mod:`.gqaw` is its ctypes binding.
"""
from .gqaw import *  # noqa: F401,F403
from .gqaw import load, make_args, new_workspace, check, GqawError  # noqa: F401
