"""fp64 CPU oracle of the mixed sliding/global attention step -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package. The product library (``mixed_sliding_global_gb300``) never imports it,
and this package imports nothing from the product.
"""
from .oracle import (  # noqa: F401
    Oracle, build_oracle, load_oracle, oracle_layers, OracleError,
)
