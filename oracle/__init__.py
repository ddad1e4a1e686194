"""Float64 CPU oracle for DDTree verify attention — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The CUDA library never calls it and
has no CPU fallback to it.  It shares no code with the CUDA path.
"""
from .verify_oracle import (  # noqa: F401
    ancestor_sets, ancestor_mask, ancestor_bits, key_mask, verify_request,
    verify_batched, partial_over_keys, merge_partials,
)
from .accept_oracle import (  # noqa: F401
    argmax_rows, greedy_path, accept_request, accept_batched,
)
from .relocate_oracle import relocate, relocation_errors  # noqa: F401
from .mask_oracle import tree_from_mask, trees_from_flat_mask  # noqa: F401
