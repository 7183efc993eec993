"""Fused residual add + RMSNorm on the GPU against the float64 oracle.

Tolerances: fp32 |out - out*| <= 2e-5 |out*| + 1e-6; bf16 outputs are rounded
once, so |out - out*| <= 2^-8 |out*| + 1e-6, and res_out must equal x + residual
rounded to bf16 exactly (the fp32 sum of two bf16 values is exact here).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_05_gb300 import add_rmsnorm, device_status

pytestmark = pytest.mark.gpu


def _inputs(rows, width, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    t = torch.float32 if dtype == "f32" else torch.bfloat16
    x = (2 * torch.randn(rows, width, generator=g)).to(t)
    r = torch.randn(rows, width, generator=g).to(t)
    w = (1 + 0.5 * torch.randn(width, generator=g)).to(t)
    return x, r, w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_res", [False, True])
# bf16 rows of up to 8192 elements (a multiple of 8) stream through two
# shared-memory stages; the larger row counts make each CTA cycle through both.
@pytest.mark.parametrize("rows,width", [(1, 1), (3, 7), (33, 8), (300, 100), (64, 512),
                                        (16, 4096), (8, 8192), (5, 8200), (3, 20000),
                                        (3000, 1024), (2000, 8192)])
def test_add_rmsnorm_parity(dtype, with_res, rows, width):
    x, r, w = _inputs(rows, width, dtype, seed=rows * 31 + width)
    eps = 1e-6
    res = r.cuda() if with_res else None
    got = add_rmsnorm(x.cuda(), w.cuda(), res, eps)
    torch.cuda.synchronize()
    assert device_status() == 0
    out, h = got if with_res else (got, None)
    ref, h_ref = oracle.add_rmsnorm(x, r if with_res else None, w, eps)
    o = out.float().cpu().numpy().astype(np.float64)
    rtol = 2e-5 if dtype == "f32" else 2.0 ** -8
    assert np.all(np.abs(o - ref) <= rtol * np.abs(ref) + 1e-6), np.abs(o - ref).max()
    if with_res:
        want = torch.from_numpy(h_ref).to(x.dtype)
        assert torch.equal(h.cpu(), want)


def test_add_rmsnorm_rejects_bad_arguments():
    x = torch.zeros(4, 8, device="cuda")
    with pytest.raises(ValueError):
        add_rmsnorm(x, torch.ones(7, device="cuda"))
    with pytest.raises(ValueError):
        add_rmsnorm(x, torch.ones(8, device="cuda", dtype=torch.bfloat16))
