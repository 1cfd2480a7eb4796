"""Exact IO-aware attention forward for GB300 (sm_103a).

The compute path is the C-ABI library libattn.so (hand-written CUDA kernels
under csrc/); this package is its thin ctypes binding plus the seeded input
generator and the work counter the benchmark uses.
"""
