"""Double-precision CPU oracle for the row-wise reduce-then-normalise operations.

Test infrastructure only: the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import it; the CUDA product path never does.
"""
