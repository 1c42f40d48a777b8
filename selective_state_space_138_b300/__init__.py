"""B300-native Mamba selective scan (S6) and single-token state update.

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI
(``include/ss_scan.h``); ``selective_state_space_138_b300.binding`` marshals
torch tensors into that ABI.
"""
__all__ = ["binding", "inputs"]
