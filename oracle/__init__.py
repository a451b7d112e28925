"""CPU float64 oracle for the dropless-MoE hot path.

TEST INFRASTRUCTURE ONLY: ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product package
never imports it, and it imports nothing from the product package; the two
share only the seeded input generators in ``ragged_grouped_gemm_topk_gb300.workloads``,
which hold none of the method's arithmetic.
"""

from . import moe, mxfp8  # noqa: F401
