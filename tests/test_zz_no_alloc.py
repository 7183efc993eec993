"""attn_fwd_noalloc: the entry point for callers that must not allocate.

Some callers of this library cannot let it call cudaMalloc: a server whose own
allocator owns all of the GPU's memory, or code running where a device
allocation is forbidden or would synchronise the device.  For them
attn_fwd_noalloc keeps its scratch (the kernels' status word) in a static
device array instead of memory obtained with cudaMalloc.  This test calls it
through the C ABI twice in a row, on different inputs, and checks each result
against attn_fwd's on the same inputs, within the tolerances the parity tests
use (bf16: 2e-2 on O, 1e-3 on LSE; fp32: 1e-5 * max|V| + 1e-5 * |o|).

The file is named so that pytest collects it last.
"""
import ctypes
import math

import pytest
import torch

from attention_attn_fwd_05_gb300 import attn_fwd, binding
from attention_attn_fwd_05_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def _noalloc(q, k, v, o, lse, causal, dtype_code):
    B, H, N, d = q.shape
    return binding.lib().attn_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
        ctypes.c_float(1.0 / math.sqrt(d)), int(causal), dtype_code,
        torch.cuda.current_stream().cuda_stream)


def _close(dtype, o, lse, o_ref, lse_ref, v):
    if dtype == "bf16":
        assert (o.float() - o_ref.float()).abs().max().item() <= 2e-2
        assert (lse - lse_ref).abs().max().item() <= 1e-3
    else:
        vmax = v.abs().max().item()
        tol = 1e-5 * vmax + 1e-5 * o_ref.abs()
        assert bool(((o - o_ref).abs() <= tol).all())
        assert bool(((lse - lse_ref).abs() <= 2e-5 + 1e-5 * lse_ref.abs()).all())


@pytest.mark.parametrize("dtype,d,causal,N", [("bf16", 128, True, 300), ("bf16", 64, False, 1000),
                                              ("f32", 64, True, 257)])
def test_noalloc_matches_attn_fwd_twice(dtype, d, causal, N):
    code = binding.ATTN_BF16 if dtype == "bf16" else binding.ATTN_F32
    for call, seed in enumerate((101, 202)):  # two calls in a row, different inputs
        q, k, v = (t.cuda() for t in make_qkv(2, 2, N, d, seed=seed + N, dtype=dtype))
        o_ref, lse_ref = attn_fwd(q, k, v, causal=causal)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((2, 2, N), float("nan"), device="cuda")
        assert _noalloc(q, k, v, o, lse, causal, code) == 0, f"call {call}"
        torch.cuda.synchronize()
        _close(dtype, o, lse, o_ref, lse_ref, v)


def test_noalloc_rejects_like_attn_fwd():
    L = binding.lib()
    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.attn_fwd_noalloc(None, x.data_ptr(), x.data_ptr(), x.data_ptr(), None, 1, 1, 128,
                              64, ctypes.c_float(0.125), 0, 1, s) == 1
    assert L.attn_fwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None, 1,
                              1, 128, 96, ctypes.c_float(0.125), 0, 1, s) == 4
    host = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    assert L.attn_fwd_noalloc(host.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None, 1,
                              1, 128, 64, ctypes.c_float(0.125), 0, 1, s) == 9
