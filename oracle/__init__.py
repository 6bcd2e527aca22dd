"""fp64 CPU oracle for the fused attention forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports, calls or links anything here, and this
package imports nothing from the product path.
"""
from .sdpa import (  # noqa: F401
    attention,
    attention_bruteforce,
    attention_varlen,
    decode,
    split_partials,
    merge_max_sum,
    merge_sequential,
    merge_lse,
    valid_key_matrix,
)
