"""Paged variable-length attention forward for NVIDIA GB300 (sm_103a).

The compute lives in the C-ABI library ``libpva.so`` (hand-written CUDA);
``paged_variable_length_gb300.pva`` is its thin ctypes binding.  Importing this
package loads nothing; the library is loaded on first use and a missing or
unbuilt library raises instead of falling back to anything else.
"""
__all__ = ["pva", "workloads"]
