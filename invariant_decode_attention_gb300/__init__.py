"""Batch-invariant split-KV decode attention for GB300 (sm_103a).

Importing the package loads nothing; the CUDA library is opened on first use
by ``invariant_decode_attention_gb300.api`` and an import error is raised
there if it has not been built.
"""

__all__ = ["api", "workloads"]
