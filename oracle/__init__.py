"""Float64 CPU oracle for the calibration Hessian.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library itself.
"""

from .hessian_oracle import (  # noqa: F401
    GramOracle,
    LocalGramOracle,
    column_sum_of_squares,
    gram_columns,
)
