"""GB300-native accumulation of the GPTQ/QQQ calibration Hessian.

``H = (2/N) sum_t x_t x_t^T`` over ragged batches of layer-input activations
(N counts tokens), damped by ``damp_percent * mean(diag H)`` when it is
materialized, plus the batched 16x16 per-block "local Hessian", and the
quantization pass that consumes H (``GPTQ``).  All of the arithmetic runs in
the CUDA library ``libgptq_hess.so`` (sm_103a) behind the C ABI in
``include/hess.h`` and ``include/gptq.h``; this package only marshals
arguments.
"""

from .hessian import *  # noqa: F401,F403
from .hessian import Hessian, IMatrix, LocalHessian  # noqa: F401
from .gptq import GPTQ  # noqa: F401
