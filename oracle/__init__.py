"""fp64 CPU oracle for kernelized linear attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library
and imports nothing from it.

Pinned functions (each checked in ``tests/test_oracle.py`` against something
other than itself: a hand-derived worked example, closed forms, invariants,
brute force, the degree-2 polynomial special case, or central finite
differences): elu_plus_one, elu_plus_one_grad, masked_attention,
masked_attention_rows, linearized_attention, recurrent_attention, forward, prefill, decode_step,
backward, denominators, poly2_feature, random_fourier_feature. No function here is parity
unpinned.
"""

from .linear_attention import (  # noqa: F401
    backward,
    decode_step,
    denominators,
    elu_plus_one,
    elu_plus_one_grad,
    forward,
    linearized_attention,
    masked_attention,
    masked_attention_rows,
    poly2_feature,
    prefill,
    random_fourier_feature,
    recurrent_attention,
)
