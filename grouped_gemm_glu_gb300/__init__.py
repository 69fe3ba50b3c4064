"""GB300-native fused MoE grouped GEMM + GLU + MXFP8/NVFP4 library.

The compute path is the C-ABI shared library ``libmoeglu.so`` (CUDA for
sm_103a) declared in ``include/moeglu.h``; ``grouped_gemm_glu_gb300.ops``
marshals torch tensors into it.  Importing this package does not load the
library; ``grouped_gemm_glu_gb300.lib.load()`` does, and raises if it is
missing.
"""
__all__ = ["synth", "lib", "ops"]
