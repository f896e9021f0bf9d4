"""GB300 (sm_103a) low-precision MoE routed-expert layer: a C-ABI CUDA
library (``libmgq.so``) and its thin Python binding (``fp8_grouped_gemm_gb300.mgq``).

Importing the package does not load the library; ``fp8_grouped_gemm_gb300.mgq``
does, and raises if it is missing.
"""
