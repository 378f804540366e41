"""Float64 CPU oracle for the Kronecker-factored optimizer step.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke entry
and by the benchmark's CPU-baseline leg; never by the library itself.
"""
from .kfac_oracle import *  # noqa: F401,F403
from .kfac_oracle import NotPositiveDefinite, KfacOracle, LayerState  # noqa: F401
