"""Exact IO-aware attention (tiled forward with online softmax, recompute
backward, block-sparse tile skipping) for NVIDIA GB300 / sm_103a.

The compute path is the CUDA library ``libfa_gb300.so`` built from ``csrc/``;
``exact_io_aware_tma_gb300.fa`` is its thin ctypes binding.  Importing this
package does not load the library; the first call into ``fa`` does, and raises
if it is missing.
"""

__all__ = ["fa", "workloads"]
