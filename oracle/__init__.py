"""Float64 CPU oracle of the KL distillation loss against a cached teacher top-K.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import it.  It shares no code with the CUDA
library.  See ``oracle/dense_kl.py`` for the definition it implements and its sources.
"""
from . import divergences  # noqa: F401
from .topk_cache import logits_at, teacher_topk  # noqa: F401
from .dense_kl import (  # noqa: F401
    backward,
    dH_rows,
    dW_rows,
    forward,
    teacher_probs,
    to_f64,
    token_weights,
)
