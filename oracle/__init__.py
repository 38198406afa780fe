"""Float64 CPU oracle for Top-theta attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path.
"""
from .topt_ref import *  # noqa: F401,F403
