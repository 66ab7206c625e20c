"""Double-precision CPU oracle for the per-token softmax divergences.

Test infrastructure only: the test suite, the smoke check and the benchmark's
CPU-baseline leg may use it; the product path never does.
"""
