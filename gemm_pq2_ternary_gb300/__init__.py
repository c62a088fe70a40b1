"""GB300 (sm_103a) PQ2_0 ternary-weight matmul.

The product is the CUDA library libpq2.so behind the C ABI of include/pq2.h.
``gemm_pq2_ternary_gb300.binding`` is its thin Python binding (same names as
the C entry points); ``gemm_pq2_ternary_gb300.inputs`` draws seeded synthetic
inputs.  Build with ``gemm_pq2_ternary_gb300._build.build()``.
"""
__version__ = "0.1"
