"""fp64 CPU oracle for the masked / biased attention path.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke check
and the benchmark's CPU-baseline leg, never by the product path.
"""
