"""Implicit-GEMM conv2d for GB300 (sm_103a)."""
