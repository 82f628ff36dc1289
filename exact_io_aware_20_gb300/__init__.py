"""Exact IO-aware attention (FlashAttention-2 class) for GB300 / sm_103a.

The compute path is the C-ABI library ``libfa_gb300.so`` built from
``csrc/``; ``binding`` marshals torch tensors into its entry points.
"""
