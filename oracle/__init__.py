"""The oracle: plain CPU definitions of the three fused operators.

TEST INFRASTRUCTURE ONLY -- imported by the tests, the smoke check and the
benchmark's CPU-baseline leg; never by the CUDA product path.
"""
