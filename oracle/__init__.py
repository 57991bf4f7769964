"""CPU oracle of the quantized GEMM / conv path.  TEST INFRASTRUCTURE ONLY:
only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg use it."""
