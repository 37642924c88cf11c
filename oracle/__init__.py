"""CPU float64 oracle for the routed / latent MoE layer forward.

This package is test infrastructure.  Only the tests, the smoke check and the
CPU-baseline leg of the benchmark may import it; the product path never does.
"""
