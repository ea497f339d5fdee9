"""GB300-native TurboQuant online KV-cache quantization.

The compute path lives in the CUDA library ``libtq.so`` (C ABI, declared in
``include/tq.h``); ``binding`` marshals arguments to it with ctypes. The
library is loaded on first use and its absence is an error: there is no CPU
fallback.
"""

__all__ = ["binding", "workloads"]
