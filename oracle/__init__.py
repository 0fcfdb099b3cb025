"""CPU oracle for the fused (add +) RMSNorm + group activation quantisation.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this package. It shares no code with
the CUDA path; the plain-C definition lives in ``rmsq_oracle.c`` and
``oracle.oracle`` wraps it with numpy arrays.
"""
