"""MLA latent-KV decode with matrix absorption, native to GB300 (sm_103a).

The compute path lives in ``libmla_gb300.so`` (hand-written CUDA behind a C ABI declared in
``include/mla.h``); ``binding`` marshals torch tensors into those calls.  ``synth`` draws the
seeded synthetic inputs.  Importing this package loads nothing; the library is opened on
first use and a missing build raises instead of falling back to anything else.
"""
from __future__ import annotations

NUM_HEADS = 128
D_HC = 128
D_C = 512
D_R = 64
D_ROW = 576
PAGE = 64

__all__ = ["NUM_HEADS", "D_HC", "D_C", "D_R", "D_ROW", "PAGE"]
