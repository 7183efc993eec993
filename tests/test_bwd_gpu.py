"""Attention backward on the GPU against the float64 oracle backward.

Both sides get the same Q, K, V, dO and the same forward outputs (O rounded to
the tensor dtype, LSE in fp32, both from the oracle forward), so the check
isolates the backward.  Tolerances (derived from fp32 accumulation over up to
N terms and, for bf16, one rounding of each output), with M = max(max|g*|, T)
where T bounds one term of the sum (scale * max|K| * 2 max|dO| max|V| for dQ,
the same with Q for dK, max|dO| for dV), so that gradients that vanish in
exact arithmetic (a single key) still get the rounding of their terms:
  fp32: |g - g*| <= 1e-4 * M + 1e-4 * |g*|
  bf16: |g - g*| <= 2e-3 * M + 2^-8 * |g*|
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_05_gb300 import attention, attn_bwd, device_status
from attention_attn_fwd_05_gb300.inputs import make_qkv, torch_dtype

pytestmark = pytest.mark.gpu


def _check(dtype, got, ref, name, term):
    g = got.float().cpu().numpy().astype(np.float64)
    m = max(np.abs(ref).max(), term)
    if dtype == "f32":
        tol = 1e-4 * m + 1e-4 * np.abs(ref)
    else:
        tol = 2e-3 * m + 2.0 ** -8 * np.abs(ref)
    bad = np.abs(g - ref) > tol
    assert not bad.any(), f"{name}: {bad.sum()} out of tolerance, max err {np.abs(g - ref).max():.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 3, 129, 300])
def test_bwd_parity(dtype, d, causal, N):
    q, k, v = make_qkv(1, 2, N, d, seed=600 + N + d, dtype=dtype)
    scale = float(torch.tensor(1 / math.sqrt(d), dtype=torch.float32))
    o64, lse64 = oracle.attn_fwd(q, k, v, scale, causal)
    t = torch_dtype(dtype)
    o = torch.from_numpy(o64).to(t)
    lse = torch.from_numpy(lse64).float()
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(N)).to(t)
    dq, dk, dv = attn_bwd(q.cuda(), k.cuda(), v.cuda(), o.cuda(), lse.cuda(), g.cuda(), scale,
                          causal)
    torch.cuda.synchronize()
    assert device_status() == 0
    rq, rk, rv = oracle.attn_bwd(q, k, v, o, g, lse, scale, causal)
    mx = lambda t: float(t.float().abs().max())
    ds_bound = 2 * mx(g) * mx(v)
    _check(dtype, dq, rq, "dQ", scale * mx(k) * ds_bound)
    _check(dtype, dk, rk, "dK", scale * mx(q) * ds_bound)
    _check(dtype, dv, rv, "dV", mx(g))


def test_autograd_function_fp32():
    """attention() under autograd against float64 autograd of the library SDPA."""
    q, k, v = make_qkv(1, 2, 200, 64, seed=70, dtype="f32")
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(3))
    qd, kd, vd = (x.cuda().requires_grad_() for x in (q, k, v))
    out = attention(qd, kd, vd, causal=True)
    out.backward(g.cuda())
    q64, k64, v64 = (x.double().requires_grad_() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(q64, k64, v64, is_causal=True)
    ref.backward(g.double())
    np.testing.assert_allclose(out.detach().cpu().numpy(), ref.detach().numpy(), atol=2e-5, rtol=1e-4)
    for a, b in ((qd, q64), (kd, k64), (vd, v64)):
        np.testing.assert_allclose(a.grad.cpu().numpy(), b.grad.numpy(), atol=2e-4, rtol=1e-3)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,dist", [(700, "normal"), (1024, "normal"), (600, "stress")])
def test_bwd_parity_bf16_multiblock(d, causal, N, dist):
    """bf16 backward over several 128-row blocks on both the key and the query
    side, ragged tails, and large logits (variance-16 Q and K)."""
    q, k, v = make_qkv(1, 2, N, d, seed=900 + N + d, dtype="bf16", dist=dist)
    scale = float(torch.tensor(1 / math.sqrt(d), dtype=torch.float32))
    o64, lse64 = oracle.attn_fwd(q, k, v, scale, causal)
    o = torch.from_numpy(o64).to(torch.bfloat16)
    lse = torch.from_numpy(lse64).float()
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(N + 1)).to(torch.bfloat16)
    dq, dk, dv = attn_bwd(q.cuda(), k.cuda(), v.cuda(), o.cuda(), lse.cuda(), g.cuda(), scale,
                          causal)
    torch.cuda.synchronize()
    assert device_status() == 0
    rq, rk, rv = oracle.attn_bwd(q, k, v, o, g, lse, scale, causal)
    mx = lambda t: float(t.float().abs().max())
    ds_bound = 2 * mx(g) * mx(v)
    _check("bf16", dq, rq, "dQ", scale * mx(k) * ds_bound)
    _check("bf16", dk, rk, "dK", scale * mx(q) * ds_bound)
    _check("bf16", dv, rv, "dV", mx(g))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [2000, 2561])
def test_bwd_parity_bf16_long_rings(d, causal, N):
    """bf16 backward over 16-21 streamed blocks per CTA, so every slot of the
    streamed rings (K/V in the dQ kernel, Q/dO pairs in the dK/dV kernel) is
    reused several times through both phases of its barriers; ragged tails."""
    q, k, v = make_qkv(1, 2, N, d, seed=1300 + N + d, dtype="bf16")
    scale = float(torch.tensor(1 / math.sqrt(d), dtype=torch.float32))
    o64, lse64 = oracle.attn_fwd(q, k, v, scale, causal)
    o = torch.from_numpy(o64).to(torch.bfloat16)
    lse = torch.from_numpy(lse64).float()
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(N + 7)).to(torch.bfloat16)
    dq, dk, dv = attn_bwd(q.cuda(), k.cuda(), v.cuda(), o.cuda(), lse.cuda(), g.cuda(), scale,
                          causal)
    torch.cuda.synchronize()
    assert device_status() == 0
    rq, rk, rv = oracle.attn_bwd(q, k, v, o, g, lse, scale, causal)
    mx = lambda t: float(t.float().abs().max())
    ds_bound = 2 * mx(g) * mx(v)
    _check("bf16", dq, rq, "dQ", scale * mx(k) * ds_bound)
    _check("bf16", dk, rk, "dK", scale * mx(q) * ds_bound)
    _check("bf16", dv, rv, "dV", mx(g))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [-0.3, 0.0, 1.0])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_parity_scales(dtype, scale, d, causal):
    """Scales other than 1/sqrt(d) (the entry point accepts any finite one):
    negative, zero (dQ and dK vanish exactly, dV is the mean of dO over the
    visible queries) and 1 (peaked rows)."""
    q, k, v = make_qkv(1, 2, 300, d, seed=1700 + d, dtype=dtype)
    scale = float(torch.tensor(scale, dtype=torch.float32))
    o64, lse64 = oracle.attn_fwd(q, k, v, scale, causal)
    o = torch.from_numpy(o64).to(torch_dtype(dtype))
    lse = torch.from_numpy(lse64).float()
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(d + 3)).to(torch_dtype(dtype))
    dq, dk, dv = attn_bwd(q.cuda(), k.cuda(), v.cuda(), o.cuda(), lse.cuda(), g.cuda(), scale,
                          causal)
    torch.cuda.synchronize()
    assert device_status() == 0
    rq, rk, rv = oracle.attn_bwd(q, k, v, o, g, lse, scale, causal)
    mx = lambda t: float(t.float().abs().max())
    ds_bound = 2 * mx(g) * mx(v)
    _check(dtype, dq, rq, "dQ", abs(scale) * mx(k) * ds_bound)
    _check(dtype, dk, rk, "dK", abs(scale) * mx(q) * ds_bound)
    _check(dtype, dv, rv, "dV", mx(g))
