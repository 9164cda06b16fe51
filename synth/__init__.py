"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This package holds no arithmetic of the decoding method itself: it only draws
numbers (counter-based SplitMix64 streams and numpy PCG64 draws) and builds
model shapes, motif prompts and random trees.  The CUDA side of the same
counter-based generator lives in ``synth/synth.cu`` and must reproduce
``gen.normal``/``gen.uniform_codes``/``gen.uniform_scales`` bit for bit.
"""
from .gen import *  # noqa: F401,F403
