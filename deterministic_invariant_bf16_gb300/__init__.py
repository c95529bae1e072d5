"""Batch-invariant bf16 LLM decoding for GB300 (sm_103a).

The compute path is the C-ABI library ``libbi.so`` built from ``csrc/``
(hand-written CUDA kernels); ``binding`` wraps its entry points one for one
with ctypes.  ``synth`` draws the seeded synthetic inputs.  Importing the
package loads nothing: the library is opened on first use and a missing
library is an error, never a fallback.
"""
__all__ = ["binding", "synth"]
