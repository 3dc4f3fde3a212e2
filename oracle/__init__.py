"""CPU oracle (test infrastructure only).

Imported by the test suite, the smoke check and the benchmark's CPU-baseline
and reference legs; never by the product library.  See ``zero_oracle``.
"""
from . import zero_oracle  # noqa: F401
