"""GB300-native software-pipelined GEMM (sm_103a).

``C = alpha*A*B + beta*C`` with the next K tile's global-to-shared copy
overlapped against the current tile's multiply-accumulate through an N-stage
shared-memory ring.  The compute lives in ``libgemm.so`` (built from
``csrc/``); ``gemm`` in this package is a thin ctypes binding over its C ABI.

Importing the package does not load the CUDA library; the first call does,
and it raises if the library is missing.  There is no CPU fallback.
"""
from .workloads import (GEMM_BF16_BF16, GEMM_BF16_F32, GEMM_F16_F32, GEMM_F32,  # noqa: F401
                        WORKLOADS, Workload, make_inputs)
