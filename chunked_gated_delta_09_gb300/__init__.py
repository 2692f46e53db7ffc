"""GB300 chunked gated delta rule backward.

The backward runs in libgdrbwd.so (hand-written sm_103a CUDA behind the C ABI of include/gdr_bwd.h);
this package builds it (``build``), loads it (``_lib``) and marshals torch tensors into it (``ops``).
``inputs`` holds the seeded synthetic workloads and ``counts`` the FLOP and byte conventions.
"""
from .ops import GdrBwdPlan, chunk_indices, gdr_bwd, plan_for, problem_to_device  # noqa: F401
from ._lib import GdrError  # noqa: F401
