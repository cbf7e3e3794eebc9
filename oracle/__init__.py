"""fp64 CPU oracle of the MoE expert block (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package; the CUDA library never does.
"""
