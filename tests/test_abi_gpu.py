"""The C ABI on a GPU: pointer checks, failure detection through the bounded
wait, and the row-softmax entry point against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_05_gb300 import (attn_fwd, attn_fwd_host, binding, device_status, row_softmax,
                                         selftest_wait_timeout)
from attention_attn_fwd_05_gb300.inputs import make_qkv, make_rows

pytestmark = pytest.mark.gpu


def _raw(q, k, v, o, lse=None, d=64, dtype=1):
    B, H, N, _ = q.shape
    return binding.lib().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr() if lse is not None else None, B, H, N, d,
                                  ctypes.c_float(0.125), 0, dtype,
                                  torch.cuda.current_stream().cuda_stream)


def test_host_pointers_rejected():
    q, k, v = make_qkv(1, 1, 128, 64, 1, "bf16")
    qd = q.cuda()
    out = torch.empty_like(qd)
    assert _raw(q, qd, qd, out) == 9             # pageable host memory
    pinned = q.pin_memory()
    assert _raw(qd, pinned, qd, out) == 9        # pinned host memory
    assert _raw(qd, qd, qd, out) == 0
    torch.cuda.synchronize()
    assert device_status() == 0


def test_bounded_wait_times_out_and_context_survives():
    """A wait on a barrier nothing signals gives up and reports
    ATTN_ERR_DEVICE_TIMEOUT; the status clears and later work is correct."""
    assert selftest_wait_timeout(2_000_000) == 8
    assert device_status() == 0
    q, k, v = make_qkv(1, 2, 300, 128, 3, "bf16")
    o, lse = attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, 128 ** -0.5, True)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


# Widths that are multiples of 4 up to 12288 take the streamed kernel (many
# rows per CTA cycle through its two buffers and their phases); longer aligned
# rows, when there are few of them, a cluster of CTAs per row ((2, 70000) and
# (8, 1048576): 8 CTAs per row); the others the general kernel.
@pytest.mark.parametrize("rows,width", [(1, 1), (3, 5), (64, 1000), (8, 11264), (4, 11265),
                                        (2, 70000), (3000, 4096), (12000, 1024), (700, 12288),
                                        (2500, 8192), (50, 12292), (9000, 4), (8, 1048576)])
def test_row_softmax_parity(rows, width):
    """Row softmax (any width, including rows past 65536) against the oracle."""
    x = make_rows(rows, width, seed=rows + width, spread=6.0)
    y, lse = row_softmax(x.cuda(), return_lse=True)
    torch.cuda.synchronize()
    y_ref, lse_ref = oracle.row_softmax(x)
    yd = y.cpu().numpy().astype(np.float64)
    # fp32 exp and a sum over `width` terms: relative error well under 1e-5.
    assert np.all(np.abs(yd - y_ref) <= 1e-5 * np.abs(y_ref) + 1e-12)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-5 * max(1.0, np.abs(lse_ref).max())
    np.testing.assert_allclose(yd.sum(axis=1), 1.0, rtol=0, atol=1e-4)


@pytest.mark.parametrize("rows,width", [(5, 513), (5000, 512), (40, 20000)])
def test_row_softmax_masked_and_in_place_both_paths(rows, width):
    """-inf entries get probability 0, in place, on either kernel."""
    x = make_rows(rows, width, seed=rows + 3, spread=3.0)
    x[:, ::7] = float("-inf")
    y_ref, _ = oracle.row_softmax(torch.where(torch.isinf(x), torch.full_like(x, -1e30), x))
    xd = x.cuda()
    row_softmax(xd, out=xd)
    torch.cuda.synchronize()
    yd = xd.cpu().numpy().astype(np.float64)
    assert (yd[:, ::7] == 0).all()
    assert np.all(np.abs(yd - y_ref) <= 1e-5 * np.abs(y_ref) + 1e-12)


@pytest.mark.parametrize("width,n", [(513, 3000), (512, 3000), (20000, 3000), (70000, 8)])
def test_row_softmax_fully_masked_row(width, n):
    """A row of -inf only: every probability 0 and LSE = -inf; other rows
    unaffected (the last case runs on the cluster kernel)."""
    x = make_rows(n, width, seed=width, spread=3.0)
    x[7] = float("-inf")
    x[n - 1] = float("-inf")
    y, lse = row_softmax(x.cuda(), return_lse=True)
    torch.cuda.synchronize()
    yd, ld = y.cpu().numpy().astype(np.float64), lse.cpu().numpy()
    assert (yd[7] == 0).all() and (yd[n - 1] == 0).all()
    assert np.isneginf(ld[7]) and np.isneginf(ld[n - 1])
    keep = [i for i in range(n) if i not in (7, n - 1)]
    y_ref, lse_ref = oracle.row_softmax(x[keep])
    assert np.all(np.abs(yd[keep] - y_ref) <= 1e-5 * np.abs(y_ref) + 1e-12)
    assert np.abs(ld[keep] - lse_ref).max() <= 1e-5 * max(1.0, np.abs(lse_ref).max())


def test_row_softmax_masked_and_in_place():
    x = make_rows(5, 513, seed=9, spread=3.0)
    x[:, ::7] = float("-inf")
    y_ref, _ = oracle.row_softmax(torch.where(torch.isinf(x), torch.full_like(x, -1e30), x))
    xd = x.cuda()
    row_softmax(xd, out=xd)  # in place
    torch.cuda.synchronize()
    yd = xd.cpu().numpy().astype(np.float64)
    assert (yd[:, ::7] == 0).all()
    assert np.all(np.abs(yd - y_ref) <= 1e-5 * np.abs(y_ref) + 1e-12)


# ------------------------------------------------ attn_fwd_host (host memory) ---

@pytest.mark.parametrize("dtype,B,H,N,d,causal", [
    ("bf16", 1, 2, 300, 64, True),       # one chunk
    ("bf16", 2, 16, 2048, 128, False),   # eight chunks
    ("bf16", 1, 11, 4096, 128, True),    # two uneven chunks (5 and 6 heads)
    ("f32", 1, 8, 1024, 64, False),      # one chunk, exact fp32 kernel
    ("f32", 2, 8, 2048, 64, True),       # four chunks, exact fp32 kernel
])
def test_fwd_host_matches_device_call(dtype, B, H, N, d, causal):
    """The pipelined host-memory call against the device call on the same
    values.  A problem copied in one chunk runs the very same launch: equal
    bit for bit.  Chunks are launched on fewer heads, which can change the
    launch shape (split CTAs for small chunks) and with it the fp32 summation
    order: then both are held to the parity tolerances."""
    q, k, v = make_qkv(B, H, N, d, seed=B * 100 + H + N, dtype=dtype)
    scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    o_dev, lse_dev = attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, causal)
    torch.cuda.synchronize()
    o_dev, lse_dev = o_dev.cpu(), lse_dev.cpu()
    elt = 2 if dtype == "bf16" else 4
    one_chunk = B * H * (4 * N * d * elt + 4 * N) < (32 << 20)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    bufs = {}
    for _ in range(2):  # the second call reuses the workspace and host outputs
        o_h, lse_h = attn_fwd_host(qh, kh, vh, scale, causal, buffers=bufs)
        assert device_status() == 0
        if one_chunk:
            assert torch.equal(o_h, o_dev) and torch.equal(lse_h, lse_dev)
            continue
        do = (o_h.float() - o_dev.float()).abs()
        dl = (lse_h - lse_dev).abs().max().item()
        if dtype == "bf16":
            assert do.max().item() <= 2e-2 and dl <= 1e-3
        else:
            tol = 1e-5 * v.abs().max().item() + 1e-5 * o_dev.abs()
            assert bool((do <= tol).all()) and dl <= 2e-5 + 1e-5 * lse_dev.abs().max().item()


def test_fwd_host_pageable_inputs_and_no_lse():
    """Pageable host inputs work, and a NULL lse skips the LSE copy; O still
    matches the device call."""
    import ctypes
    from attention_attn_fwd_05_gb300.binding import lib
    B, H, N, d = 1, 4, 1000, 128
    q, k, v = make_qkv(B, H, N, d, seed=5, dtype="bf16")
    scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    o_dev, _ = attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, False)
    nbytes = lib().attn_fwd_host_workspace_bytes(B, H, N, d, 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o_h = torch.empty_like(q)  # pageable
    s = torch.cuda.current_stream()
    st = lib().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_h.data_ptr(), None,
                             B, H, N, d, ctypes.c_float(scale), 0, 1, ws.data_ptr(), nbytes,
                             s.cuda_stream)
    assert st == 0
    s.synchronize()
    assert device_status() == 0
    assert torch.equal(o_h, o_dev.cpu())


def test_fwd_host_two_calls_in_flight():
    """wait=False: two calls on two streams with their own buffers overlap, and
    each returns exactly what a waiting call returns."""
    B, H, N, d = 2, 8, 2048, 128
    # Pinned inputs held for the whole test: a call that does not wait still
    # reads them after it returns.
    probs = [tuple(t.pin_memory() for t in make_qkv(B, H, N, d, seed=s, dtype="bf16"))
             for s in (21, 22, 23, 24)]
    ref = [attn_fwd_host(*p, causal=True) for p in probs]
    ref = [(o.clone(), l.clone()) for o, l in ref]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = [{}, {}]
    outs = []
    for i, p in enumerate(probs):
        if i >= 2:
            streams[i % 2].synchronize()
            outs.append(tuple(t.clone() for t in last[i % 2]))
        res = attn_fwd_host(*p, causal=True, stream=streams[i % 2], buffers=bufs[i % 2],
                            wait=False)
        if i < 2:
            last = [None, None] if i == 0 else last
        last[i % 2] = res
    for st in streams:
        st.synchronize()
    outs += [tuple(t.clone() for t in last[0]), tuple(t.clone() for t in last[1])]
    assert device_status() == 0
    for (o, l), (o_r, l_r) in zip(outs, ref):
        assert torch.equal(o, o_r) and torch.equal(l, l_r)
