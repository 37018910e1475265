"""GB300 (sm_103a) packed weight-only-quantized decode GEMV/GEMM.

``C[M,N] = A[M,K] @ dequant(W)^T`` with BF16 activations, M = 1..16 rows and
the weights kept packed in HBM (ternary Q2_0, E2M1 + E4M3 group scales, FP8
E4M3 + FP32 128x128 block scales). Every step runs in the CUDA kernels of
``libwqp.so``; this package only marshals arguments (see ``binding``).
"""
from .binding import *  # noqa: F401,F403
from .binding import __all__  # noqa: F401
