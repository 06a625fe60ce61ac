"""Float64 CPU oracle for exact softmax attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` use this package.  The CUDA library never imports it.
"""

from .attention import (  # noqa: F401
    attention_backward,
    attention_forward,
    attention_forward_gqa,
    attention_decode_paged,
    gather_pages,
    attention_probs,
    attention_rows,
    backward_delta,
    causal_visible,
    merge_partials,
    online_attention,
    scores,
    split_partials,
)
