"""The bounds-checking debug build on the GPU.

The library's sources compiled with -DATTN_DEBUG_BOUNDS make every forward
kernel test each global index and TMA coordinate against B*H, N and d before
the access; a failed test records a status bit (attn_device_status then
returns ATTN_ERR_DEVICE_BOUNDS) and skips the access instead of trapping.  It
stands in for a memory checker on the awkward shapes: 1, 2, 3, 127, 129 and
300 rows (ragged tiles, tiles past the end), both head dims, both masks, bf16
on the split kernel alone and on the main kernel with a split tail, and fp32.
Only valid inputs are run: the status must read 0 and the outputs must match
the oracle at the parity tolerances.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_05_gb300.build import build
from attention_attn_fwd_05_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def DL():
    path = build(bounds_checks=True)
    L = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                           ctypes.c_int, ctypes.c_int, vp]
    L.attn_fwd.restype = ctypes.c_int
    L.attn_device_status.argtypes = [vp]
    L.attn_device_status.restype = ctypes.c_int
    return L


SHAPES = [(1, 1, 1), (1, 2, 2), (2, 1, 3), (1, 2, 127), (1, 1, 129), (2, 2, 300),
          (2, 40, 300), (1, 80, 129)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", SHAPES)
def test_bounds_build_reports_no_out_of_range_access(DL, dtype, d, causal, B, H, N):
    q, k, v = make_qkv(B, H, N, d, seed=4000 + N + H, dtype=dtype)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    scale = float(np.float32(1.0 / math.sqrt(d)))
    s = torch.cuda.current_stream().cuda_stream
    code = 1 if dtype == "bf16" else 0
    assert DL.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                       lse.data_ptr(), B, H, N, d, ctypes.c_float(scale), int(causal), code,
                       s) == 0
    assert DL.attn_device_status(s) == 0  # no bounds bit, no timeout
    o_ref, l_ref = oracle.attn_fwd(q, k, v, scale, causal)
    eo = np.abs(o.float().cpu().numpy() - o_ref)
    el = np.abs(lse.cpu().numpy() - l_ref)
    if dtype == "bf16":
        assert eo.max() <= 2e-2 and el.max() <= 1e-3, (eo.max(), el.max())
    else:
        vmax = float(v.abs().max())
        assert (eo <= 1e-5 * vmax + 1e-5 * np.abs(o_ref)).all(), eo.max()
        assert (el <= 2e-5 + 1e-5 * np.abs(l_ref)).all(), el.max()
