"""Float64 CPU oracle for absorbed-MLA decode -- test infrastructure only.

Importable by the tests, the smoke check and the benchmark's CPU-baseline leg.
The library never imports it.
"""
from .mla_oracle import *  # noqa: F401,F403
