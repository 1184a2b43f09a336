"""fp64 CPU oracle of the joint-sequence attention hot path.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the product path never does.
"""
