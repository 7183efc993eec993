"""attn_fwd_noalloc: the entry point for callers that must not allocate.

Some callers of this library cannot let it call cudaMalloc: a server whose own
allocator owns all of the GPU's memory, or code running where a device
allocation is forbidden or would synchronise the device.  For them
attn_fwd_noalloc keeps its scratch (the kernels' status word) in a static
device array instead of memory obtained with cudaMalloc.  This test calls it
through the C ABI twice in a row, on different inputs, and checks each result
against attn_fwd's on the same inputs, within the tolerances the parity tests
use (bf16: 2e-2 on O, 1e-3 on LSE; fp32: 1e-5 * max|V| + 1e-5 * |o|).

A second test runs in a fresh Python process that calls attn_fwd_noalloc
before anything else of the library on the device: it checks the results
against the oracle and that the device's free memory did not change across the
calls (CUDA modules are loaded eagerly in that process, so loading kernel code
does not show up as a change).  attn_fwd is never called there.

The file is named so that pytest collects it last.
"""
import ctypes
import json
import math
import os
import subprocess
import sys
import textwrap

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
        assert binding.lib().attn_fwd_noalloc_status(
            torch.cuda.current_stream().cuda_stream) == 0, f"call {call}: device timeout"
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


_FRESH = textwrap.dedent(r"""
    import ctypes, json, math, sys
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    import oracle
    from attention_attn_fwd_05_gb300 import binding
    from attention_attn_fwd_05_gb300.inputs import make_qkv

    L = binding.lib()
    cases = []
    for dtype, d, causal, N in (("bf16", 128, True, 300), ("bf16", 64, False, 700),
                                ("f32", 64, True, 257)):
        q, k, v = (t.cuda() for t in make_qkv(1, 2, N, d, seed=N, dtype=dtype))
        o = torch.full_like(q, float("nan"))
        lse = torch.full((1, 2, N), float("nan"), device="cuda")
        cases.append((dtype, d, causal, N, q, k, v, o, lse))
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    status = []
    for rep in range(2):  # every case twice in a row
        for dtype, d, causal, N, q, k, v, o, lse in cases:
            code = binding.ATTN_BF16 if dtype == "bf16" else binding.ATTN_F32
            status.append(L.attn_fwd_noalloc(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 2,
                N, d, ctypes.c_float(1.0 / math.sqrt(d)), int(causal), code, stream))
    status.append(L.attn_fwd_noalloc_status(stream))
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    errs = []  # elements outside the parity tolerances, per case
    for dtype, d, causal, N, q, k, v, o, lse in cases:
        o_ref, l_ref = oracle.attn_fwd(q.cpu(), k.cpu(), v.cpu(),
                                       float(np.float32(1.0 / math.sqrt(d))), causal)
        eo = np.abs(o.float().cpu().numpy() - o_ref)
        el = np.abs(lse.cpu().numpy() - l_ref)
        if dtype == "bf16":
            bad = int((eo > 2e-2).sum() + (el > 1e-3).sum())
        else:
            vmax = float(v.abs().max())
            bad = int((eo > 1e-5 * vmax + 1e-5 * np.abs(o_ref)).sum()
                      + (el > 2e-5 + 1e-5 * np.abs(l_ref)).sum())
        errs.append([dtype, d, causal, N, bad, float(eo.max()), float(el.max())])
    print(json.dumps({"status": status, "free0": free0, "free1": free1, "errs": errs}))
""")


def test_noalloc_first_in_a_fresh_process_allocates_nothing():
    """In a process that has never called attn_fwd, attn_fwd_noalloc (and its
    status query) work, match the oracle, and leave the device's free memory
    unchanged: nothing was allocated on the device."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True,
                       timeout=600, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert all(s == 0 for s in res["status"]), res["status"]
    assert res["free1"] == res["free0"], (res["free0"], res["free1"])
    for case in res["errs"]:
        assert case[4] == 0, case
