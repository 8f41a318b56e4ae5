"""fp64 CPU oracle for exact attention -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never does, and the
product path has no CPU fallback.
"""

from .attention import (  # noqa: F401
    backward,
    backward_preprocess,
    combine,
    effective_kv_lens,
    forward,
    probabilities,
    split_bounds,
    splitkv_partials,
    valid_keys,
)
