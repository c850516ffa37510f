"""Seeded synthetic inputs for the DSA lightning-indexer workloads.

This package generates inputs only: batch metadata (query counts, context
lengths, page tables) and the FP32 tensors a model layer would hand to the
indexer (new-token keys, cached-prefix keys, queries, head weights).  It holds
none of the indexer's arithmetic (no quantisation, no slot arithmetic, no
scoring, no selection, no layer schedule), so the CPU oracle and the CUDA
path can both consume it without sharing any step of the method.
"""

from .workloads import (  # noqa: F401
    HEAD_DIM,
    PAGE_TOKENS,
    Workload,
    make_workload,
    WORKLOAD_NAMES,
)
