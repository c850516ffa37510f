"""DSA lightning-indexer step for one GB300 GPU (sm_103a CUDA kernels, C ABI).

The compute path is ``libdsa_indexer.so`` (see include/dsa_indexer.h); the
Python modules only marshal tensors into its entry points.  Importing this
package does not load the library; the first call into :mod:`.binding` does,
and raises if it was not built (there is no CPU fallback).
"""

from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    DsaError,
    layer_is_full,
    layer_stack_run,
    quantize_fp8_blocks,
    score_topk,
    workspace_bytes,
    alloc_workspace,
    write_k,
)
