"""GB300-native chunkwise Gated DeltaNet forward with per-segment affine state summaries.

The compute path is the C-ABI library ``libgdn.so`` (hand-written sm_103a CUDA kernels);
``context_scan_gb300.gdn`` is its thin ctypes binding. Importing this package loads no
library: the binding loads ``libgdn.so`` on first use and raises if it is missing.
"""
__all__ = ["gdn", "synth"]
