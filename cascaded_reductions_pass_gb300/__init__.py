"""Fused cascaded reductions on GB300 (sm_103a): Python binding of librf.so."""
from ._binding import *  # noqa: F401,F403
from ._binding import load  # noqa: F401
