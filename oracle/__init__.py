"""fp64 CPU oracle for split-KV Flash Decode -- test infrastructure, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu-baseline and
reference legs may import this package.  The CUDA library never imports, links
or calls it, and it imports nothing from the CUDA library.

Every function is pinned by ``tests/test_oracle.py`` (``-m "not gpu"``) against
brute force, closed forms, invariants and library routines; no function here is
"parity unpinned".
"""
from .fd_oracle import (  # noqa: F401
    NEG_INF,
    combine2,
    decode_reference,
    default_scale,
    finalize,
    gather_paged,
    online_softmax_combine,
    segment_bounds,
    segment_partial,
    split_kv_decode,
    widen,
)
