"""Q8_0 W8A16 decode matmul for GB300 (sm_103a): the libq8 C ABI and its binding.

The compute path is ``libq8.so`` (hand-written CUDA, see ``csrc/``); this
package only builds it (``build.py``) and marshals arguments to it (``q8.py``).
"""
from . import q8  # noqa: F401
from .q8 import (Q8Error, q8_gemm, q8_gemm_skinny, q8_gemv, q8_linear_batch,  # noqa: F401
                 q8_quantize_rows, q8_workspace_size)
