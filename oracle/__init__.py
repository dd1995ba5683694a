"""fp64 CPU oracle of the MoE expert layer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg, never by the product path.  It shares no
code with the CUDA kernels.  Every function is pinned: ``moe_ref`` by
``tests/test_oracle.py`` (brute force on tiny inputs, hand-worked golden
fixtures, closed forms, invariants and finite differences), ``moe_fp8_ref`` by
``tests/test_oracle_fp8.py`` and ``moe_mx_ref`` by ``tests/test_oracle_mx.py``;
no function here is "parity unpinned".
"""
from . import moe_ref  # noqa: F401
