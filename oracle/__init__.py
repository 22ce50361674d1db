"""CPU oracle of the routed NVFP4 MoE expert layer (test infrastructure).

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA path.
"""
