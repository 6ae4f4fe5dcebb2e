"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or calls anything here, and this package imports
nothing from the product path.
"""
from . import dropout  # noqa: F401
from .attention import (  # noqa: F401
    visible,
    scores,
    probabilities,
    forward,
    backward,
    forward_rows,
    backward_query_rows,
    backward_key_rows,
    row_stats,
    softmax_three_pass,
    softmax_online_two_pass,
    attention_row_one_pass_tiled,
    row_block_forward_backward,
)
