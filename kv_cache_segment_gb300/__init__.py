"""Multi-Segment Attention (MSA) for GB300 (sm_103a).

The compute path lives in the C-ABI library ``libmsa.so`` (hand-written CUDA
kernels and a C++ planner, built from ``csrc/``); ``msa`` is its thin ctypes
binding.  ``workloads`` draws seeded synthetic inputs.
"""
