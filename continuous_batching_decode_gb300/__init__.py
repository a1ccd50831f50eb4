"""cbd: one iteration-level batched decode step of a GQA transformer on GB300.

The step, the KV pool and the scheduler are in libcbd.so (hand-written CUDA
for sm_103a plus a C++ host scheduler) behind the C ABI in include/cbd.h.
This package is the thin ctypes binding (``_cbd``), the in-tree build
(``build``) and the seeded synthetic inputs (``synth``).
"""
from ._cbd import *  # noqa: F401,F403
from ._cbd import CbdError, lib  # noqa: F401
