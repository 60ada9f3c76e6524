"""Q4_K x M-row weight-streaming decode matmul for one GB300 (sm_103a).

The compute path is libqmm.so (hand-written CUDA, C ABI in include/qmm.h); ``qmm`` is
its ctypes binding.  Build with ``python -m bit_weight_streaming_q4_gb300.build``.
"""
from .qmm import BACKEND_AUTO, BACKEND_MMA_SYNC, BACKEND_TCGEN05, Qmm, QmmError, Step, load

__all__ = ["Qmm", "Step", "QmmError", "load", "BACKEND_AUTO", "BACKEND_MMA_SYNC",
           "BACKEND_TCGEN05"]
