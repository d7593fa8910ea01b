"""GB300-native GDN (Gated DeltaNet) recurrent-state decode library.

The compute path is a C-ABI shared library of hand-written CUDA kernels for
sm_103a (include/gdn.h); `hybrid_ssm_gated_gb300.gdn` is its thin ctypes
binding. `hybrid_ssm_gated_gb300.workload` draws the seeded synthetic inputs.
"""
__all__ = ["gdn", "workload"]
