"""C3 on one GB300: a bf16 tcgen05 GEMM overlapped with an emulated 8-rank
all-gather / all-to-all, carried by SM copy kernels or copy engines.

Importing the package loads nothing native.  ``concurrent_communication_overlap_gb300.c3``
is the binding to the C-ABI library ``libc3.so``; it raises if the library is missing.
"""
__all__ = ["inputs"]
