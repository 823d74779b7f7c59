"""Paged MLA decode (absorbed-MQA form) for GB300 / sm_103a.

The compute path is the C-ABI library ``libmla.so`` built from ``csrc/`` (declared in
``include/mla.h``). ``api`` is a thin ctypes binding over it that takes torch tensors
for device memory and streams; ``synth`` draws seeded synthetic workloads. Importing
this package loads nothing native: the library is opened on first use of ``api`` and
a missing library raises immediately (there is no fallback path).
"""
__all__ = ["api", "synth"]
