"""GB300-native (sm_103a) exact attention forward.

O = softmax(scale * Q K^T) V plus the per-row log-sum-exp, computed by
hand-written CUDA kernels (tcgen05 tensor cores with TMEM accumulators and TMA
for bf16; exact fp32 FMA on CUDA cores for fp32) behind a C ABI
(``include/attn_fwd.h``).  This package is the thin Python binding over that
library plus the seeded input generators.
"""
from .binding import (AttnError, AttnGraph, Attention, add_rmsnorm, attention, attn_bwd,
                      attn_fwd, attn_fwd_host, device_status, lib, row_softmax,
                      selftest_wait_timeout)
from .build import build

__all__ = ["AttnError", "AttnGraph", "Attention", "add_rmsnorm", "attention", "attn_bwd", "attn_fwd", "attn_fwd_host", "device_status",
           "lib", "row_softmax", "selftest_wait_timeout", "build"]
