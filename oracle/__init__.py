"""CPU oracle for the Q8_0 block-quantized linear layer.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports or calls it.
"""
