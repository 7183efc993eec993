"""GPU parity: the CUDA library against the float64 oracle, through the C ABI.

Tolerances (elementwise):
  fp32 path:  |o - o*| <= 1e-5 * max|V| + 1e-5 * |o*|
              |lse - lse*| <= 2e-5 + 1e-5 * |lse*|
  bf16 path:  max |o - o*| <= 2e-2 and max |lse - lse*| <= 1e-3
The oracle sees exactly the values the GPU sees (bf16 widened to float32).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_05_gb300 import attn_fwd, device_status, inputs
from attention_attn_fwd_05_gb300.inputs import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu

F32_ATOL_V, F32_RTOL = 1e-5, 1e-5
F32_LSE_ATOL, F32_LSE_RTOL = 2e-5, 1e-5
BF16_O_ATOL, BF16_LSE_ATOL = 2e-2, 1e-3


def _scale(d):
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def assert_close(dtype, o, lse, o_ref, lse_ref, vmax, what=""):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{what}: non-finite output"
    if dtype == "f32":
        tol = F32_ATOL_V * vmax + F32_RTOL * np.abs(o_ref)
        bad = np.abs(o - o_ref) > tol
        assert not bad.any(), (f"{what}: {bad.sum()} O elements out of tolerance, max err "
                               f"{np.abs(o - o_ref).max():.3e}")
        ltol = F32_LSE_ATOL + F32_LSE_RTOL * np.abs(lse_ref)
        lbad = np.abs(lse - lse_ref) > ltol
        assert not lbad.any(), f"{what}: LSE max err {np.abs(lse - lse_ref).max():.3e}"
    else:
        eo = np.abs(o - o_ref).max()
        el = np.abs(lse - lse_ref).max()
        assert eo <= BF16_O_ATOL, f"{what}: O max abs err {eo:.3e}"
        assert el <= BF16_LSE_ATOL, f"{what}: LSE max abs err {el:.3e}"


def run_gpu(q, k, v, scale, causal):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn_fwd(qd, kd, vd, scale, causal)
    torch.cuda.synchronize()
    assert device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


# --------------------------------------------------- small, full oracle ---

SMALL_SHAPES = [
    (1, 1, 1), (1, 1, 2), (1, 2, 3), (2, 1, 127), (1, 2, 128), (1, 1, 129),
    (1, 1, 256), (1, 1, 257), (1, 2, 384), (2, 2, 300), (1, 3, 513), (1, 1, 1000),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", SMALL_SHAPES)
def test_parity_small(dtype, d, causal, B, H, N):
    q, k, v = make_qkv(B, H, N, d, seed=1000 + N + d, dtype=dtype)
    scale = _scale(d)
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close(dtype, o, lse, o_ref, lse_ref, float(v.float().abs().max()),
                 f"{dtype} d={d} causal={causal} {B}x{H}x{N}")


# Small grids (at most half as many 256-row items as SMs) run entirely on the
# split kernel (two CTAs per item, key tiles split between the two query
# tiles), so the shapes above exercise it.  These shapes have more items than
# that: the main kernel runs, and without the causal mask the items of a last
# wave that would be at most half full go to the split kernel after it.
MIXED_SHAPES = [(2, 40, 300), (1, 80, 129), (1, 160, 40)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", MIXED_SHAPES)
def test_parity_main_kernel_and_tail(d, causal, B, H, N):
    q, k, v = make_qkv(B, H, N, d, seed=2000 + N + d + H, dtype="bf16")
    scale = _scale(d)
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close("bf16", o, lse, o_ref, lse_ref, float(v.float().abs().max()),
                 f"bf16 d={d} causal={causal} {B}x{H}x{N}")


# All-split grids with long key loops: every item goes to the split kernel
# (at most half as many items as SMs), and each of its query tiles walks 8 or
# more key tiles, so its barriers go through many phases (ragged N included).
SPLIT_LONG_SHAPES = [(1, 4, 4096), (2, 1, 3001)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", SPLIT_LONG_SHAPES)
def test_parity_split_long_key_loops(d, causal, B, H, N):
    q, k, v = make_qkv(B, H, N, d, seed=7000 + N + d + H, dtype="bf16")
    scale = _scale(d)
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close("bf16", o, lse, o_ref, lse_ref, float(v.float().abs().max()),
                 f"bf16 d={d} causal={causal} {B}x{H}x{N}")


# Grids of two to three waves of 256-row items on the main kernel: CTAs of
# one SM run items of different lengths (causal) one after the other, with
# ragged last tiles, both head dims and items of different heads.
MULTI_WAVE_SHAPES = [(1, 200, 300), (3, 70, 257), (2, 100, 129), (1, 160, 700)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", MULTI_WAVE_SHAPES)
def test_parity_multi_wave(d, causal, B, H, N):
    q, k, v = make_qkv(B, H, N, d, seed=5000 + N + d + H, dtype="bf16")
    scale = _scale(d)
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close("bf16", o, lse, o_ref, lse_ref, float(v.float().abs().max()),
                 f"bf16 d={d} causal={causal} {B}x{H}x{N}")


@pytest.mark.parametrize("scale", [-0.3, 0.0, 1.0])
def test_parity_multi_wave_scales_stress(scale):
    q, k, v = make_qkv(1, 160, 700, 128, seed=5100, dtype="bf16", dist="stress")
    o, lse = run_gpu(q, k, v, scale, True)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, True)
    assert_close("bf16", o, lse, o_ref, lse_ref, 1.0, f"multi-wave stress scale={scale}")


def test_multi_wave_deterministic_and_lse_optional():
    q, k, v = make_qkv(2, 100, 513, 128, seed=5200, dtype="bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = attn_fwd(qd, kd, vd, causal=True)
    o2, l2 = attn_fwd(qd, kd, vd, causal=True)
    o3, l3 = attn_fwd(qd, kd, vd, causal=True, return_lse=False)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3) and l3 is None


@pytest.mark.parametrize("causal", [False, True])
def test_parity_stress_logits_small(causal):
    """Large logits (variance-16 Q and K) on a ragged size: online-softmax stability."""
    q, k, v = make_qkv(1, 2, 700, 128, seed=77, dtype="bf16", dist="stress")
    scale = _scale(128)
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close("bf16", o, lse, o_ref, lse_ref, 1.0, "stress")


# ------------------------------------------------ scales other than 1/sqrt(d) ---
#
# The bf16 kernels take each row's maximum of the raw logits and multiply it by
# the base-2 scale, so the sign of the scale matters (a negative scale is
# folded into the S product); a zero scale must not turn masked logits into
# NaN.  Every path is covered: the split kernel alone (small grids), the main
# kernel with a split tail, d = 64 and 128, both masks, plain and stress
# (variance-16) inputs.

SCALES = [0.05, 0.3, 1.0, -0.3, "-1/sqrt(d)", 0.0]


def _resolve(scale, d):
    if scale == "-1/sqrt(d)":
        return -_scale(d)
    return float(torch.tensor(scale, dtype=torch.float32))


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,dist", [(1, 2, 700, "stress"), (2, 40, 300, "normal")])
def test_parity_scales_bf16(scale, d, causal, B, H, N, dist):
    q, k, v = make_qkv(B, H, N, d, seed=3000 + N + d, dtype="bf16", dist=dist)
    sc = _resolve(scale, d)
    o, lse = run_gpu(q, k, v, sc, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, sc, causal)
    assert_close("bf16", o, lse, o_ref, lse_ref, float(v.float().abs().max()),
                 f"bf16 d={d} causal={causal} scale={sc} {B}x{H}x{N} {dist}")


@pytest.mark.parametrize("scale", [1.0, -0.3, 0.0])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_parity_scales_f32(scale, d, causal):
    q, k, v = make_qkv(1, 3, 333, d, seed=3100 + d, dtype="f32")
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close("f32", o, lse, o_ref, lse_ref, float(v.abs().max()),
                 f"f32 d={d} causal={causal} scale={scale}")


@pytest.mark.parametrize("scale", ["-1/sqrt(d)", 0.3])
def test_parity_scales_stress_workload_size(scale):
    """The variance-16 stress shape at full size (B=2 H=16 N=4000 d=128,
    causal) with a negative and a larger positive scale, on sampled rows of
    every head plus the whole last tile."""
    w = WORKLOADS["bf16_B2_H16_N4000_d128_causal_stress"]
    q, k, v = inputs.make_workload_inputs(w)
    sc = _resolve(scale, w.d)
    o, lse = run_gpu(q, k, v, sc, w.causal)
    rng = np.random.default_rng(w.seed + 1)
    rows = _sample_rows(w, rng)
    BH = w.B * w.H
    bh_idx = np.repeat(np.arange(BH), len(rows))
    row_idx = np.tile(np.array(rows), BH)
    tail = np.arange(w.N - 128, w.N)
    bh_idx = np.concatenate([bh_idx, np.full(tail.shape, BH - 1)])
    row_idx = np.concatenate([row_idx, tail])
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, v, sc, w.causal, bh_idx, row_idx)
    of = o.reshape(BH, w.N, w.d)[bh_idx, row_idx]
    lf = lse.reshape(BH, w.N)[bh_idx, row_idx]
    assert_close("bf16", of, lf, o_ref, lse_ref, 1.0, f"stress workload scale={sc}")


def test_negative_scale_equals_negated_queries_bitwise():
    """scale < 0 on Q equals |scale| on -Q bit for bit: the kernel folds the
    sign into the S product, and negating bf16 operands is exact."""
    q, k, v = make_qkv(2, 8, 1000, 128, seed=3200, dtype="bf16", dist="stress")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    sc = _scale(128)
    o1, l1 = attn_fwd(qd, kd, vd, -sc, True)
    o2, l2 = attn_fwd((-qd).contiguous(), kd, vd, sc, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional():
    q, k, v = make_qkv(1, 1, 200, 64, seed=5, dtype="bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, _ = attn_fwd(qd, kd, vd, causal=True)
    o2, lse = attn_fwd(qd, kd, vd, causal=True, return_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    assert torch.equal(o1, o2)


# ------------------------------------------------ the named workloads ---

def _sample_rows(w, rng):
    """Rows checked per workload: tile edges, the ragged tail, random rows."""
    N = w.N
    base = {0, 1, 63, 64, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1}
    base |= set(rng.integers(0, N, size=24).tolist())
    return sorted(r for r in base if 0 <= r < N)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_parity_workload(name):
    """Every named workload at full size, in the launch configuration the bench
    times: all outputs against the oracle where it is cheap, else sampled rows
    of every head (plus one whole last tile)."""
    w = WORKLOADS[name]
    q, k, v = inputs.make_workload_inputs(w)
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    vmax = float(v.float().abs().max())
    if w.B * w.H * w.N * w.N * w.d <= 2 ** 33:
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.scale, w.causal)
        _report(name, "all rows", o, lse, o_ref, lse_ref)
        assert_close(w.dtype, o, lse, o_ref, lse_ref, vmax, name)
        return
    rng = np.random.default_rng(w.seed)
    BH = w.B * w.H
    rows = _sample_rows(w, rng)
    bh_idx = np.repeat(np.arange(BH), len(rows))
    row_idx = np.tile(np.array(rows), BH)
    tail = np.arange(max(0, w.N - 128), w.N)  # one whole last tile of the last head
    bh_idx = np.concatenate([bh_idx, np.full(tail.shape, BH - 1)])
    row_idx = np.concatenate([row_idx, tail])
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, v, w.scale, w.causal, bh_idx, row_idx)
    of = o.reshape(BH, w.N, w.d)[bh_idx, row_idx]
    lf = lse.reshape(BH, w.N)[bh_idx, row_idx]
    _report(name, f"{len(row_idx)} sampled rows", of, lf, o_ref, lse_ref)
    assert_close(w.dtype, of, lf, o_ref, lse_ref, vmax, name)


def _report(name, rows, o, lse, o_ref, lse_ref):
    """One line per workload with the measured errors (shown with pytest -s)."""
    eo = float(np.abs(np.asarray(o, np.float64) - o_ref).max())
    el = float(np.abs(np.asarray(lse, np.float64) - lse_ref).max())
    print(f"\nPARITY {name} ({rows}): max|O-O*| {eo:.2e}, max|LSE-LSE*| {el:.2e}")


@pytest.mark.parametrize("causal", [True, False])
def test_parity_head_groups_with_partial_last_group(causal):
    """B=1 H=11 N=16384 d=128: K and V of all heads exceed 64 MB, so heads are
    dispatched in groups of 8 and 3 (every item of the partial group, every
    head and the tile edges checked on sampled rows, plus whole tiles at the
    start and end of the last head)."""
    B, H, N, d = 1, 11, 16384, 128
    q, k, v = make_qkv(B, H, N, d, seed=77, dtype="bf16")
    scale = _scale(d)
    o, lse = run_gpu(q, k, v, scale, causal)
    rng = np.random.default_rng(77)
    rows = sorted({0, 1, 127, 128, 255, 256, 257, 8191, 8192, N - 129, N - 128, N - 1}
                  | set(rng.integers(0, N, size=12).tolist()))
    bh_idx = np.repeat(np.arange(B * H), len(rows))
    row_idx = np.tile(np.array(rows), B * H)
    edge = np.concatenate([np.arange(0, 128), np.arange(N - 128, N)])
    bh_idx = np.concatenate([bh_idx, np.full(edge.shape, B * H - 1)])
    row_idx = np.concatenate([row_idx, edge])
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, v, scale, causal, bh_idx, row_idx)
    of = o.reshape(B * H, N, d)[bh_idx, row_idx]
    lf = lse.reshape(B * H, N)[bh_idx, row_idx]
    assert_close("bf16", of, lf, o_ref, lse_ref, float(v.float().abs().max()),
                 f"H=11 N=16384 causal={causal}")


# ------------------------------------------------------ large extents ---

def test_parity_long_sequence_sampled_rows():
    """N = 131072 (d = 64, causal): row and key-tile coordinates far beyond the
    named workloads, checked on sampled rows of both heads, the first and last
    tiles whole."""
    B, H, N, d = 1, 2, 131072, 64
    q, k, v = make_qkv(B, H, N, d, seed=91, dtype="bf16")
    scale = _scale(d)
    o, lse = run_gpu(q, k, v, scale, True)
    rng = np.random.default_rng(91)
    rows = sorted({0, 1, 127, 128, 65535, 65536, N - 129, N - 128, N - 1}
                  | set(rng.integers(0, N, size=16).tolist()))
    bh_idx = np.repeat(np.arange(B * H), len(rows))
    row_idx = np.tile(np.array(rows), B * H)
    edge = np.concatenate([np.arange(0, 128), np.arange(N - 128, N)])
    bh_idx = np.concatenate([bh_idx, np.full(edge.shape, B * H - 1)])
    row_idx = np.concatenate([row_idx, edge])
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, v, scale, True, bh_idx, row_idx)
    of = o.reshape(B * H, N, d)[bh_idx, row_idx]
    lf = lse.reshape(B * H, N)[bh_idx, row_idx]
    assert_close("bf16", of, lf, o_ref, lse_ref, float(v.float().abs().max()), "N=131072")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_parity_many_heads(dtype):
    """B*H = 4096 heads of 130 rows: a grid of many waves (bf16: 4096 items) and
    the last head's ragged tile, against the oracle on every row."""
    q, k, v = make_qkv(64, 64, 130, 64, seed=92, dtype=dtype)
    scale = _scale(64)
    o, lse = run_gpu(q, k, v, scale, False)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, False)
    assert_close(dtype, o, lse, o_ref, lse_ref, float(v.float().abs().max()), f"{dtype} B*H=4096")


@pytest.mark.parametrize("causal", [False, True])
def test_parity_heads_beyond_65535_bf16(causal):
    """B*H = 70000 heads of 3 rows (bf16): item indices of the kernels' 1-D grid
    past 65535, against the oracle on every row.  (The exact-fp32 path keeps
    B*H <= 65535.)"""
    q, k, v = make_qkv(7, 10000, 3, 64, seed=93, dtype="bf16")
    scale = _scale(64)
    o, lse = run_gpu(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    assert_close("bf16", o, lse, o_ref, lse_ref, float(v.float().abs().max()), "B*H=70000")


# --------------------------------------------------- GPU invariances ---

def test_t3g_key_shift_on_gpu():
    """K' = K + 1 u^T: O unchanged, LSE shifted by scale * q.u (fp32, exact inputs)."""
    q, k, v = make_qkv(1, 2, 300, 64, seed=31, dtype="f32")
    u = (torch.arange(64) % 8).float() / 4 - 1  # multiples of 1/4: K + u stays exact
    k = torch.round(k * 64) / 64
    k2 = k + u
    assert torch.equal(k2 - u, k)
    scale = _scale(64)
    o1, l1 = run_gpu(q, k, v, scale, True)
    o2, l2 = run_gpu(q, k2, v, scale, True)
    np.testing.assert_allclose(o2, o1, rtol=1e-4, atol=2e-5)
    shift = (scale * (q.double() @ u.double())).numpy()
    np.testing.assert_allclose(l2, l1 + shift, rtol=1e-5, atol=5e-5)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_t4g_permutation_on_gpu(dtype):
    """Permuting K and V rows together (non-causal) leaves O and LSE unchanged."""
    q, k, v = make_qkv(1, 2, 333, 128, seed=32, dtype=dtype)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(333))
    o1, l1 = run_gpu(q, k, v, _scale(128), False)
    o2, l2 = run_gpu(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), _scale(128),
                     False)
    if dtype == "f32":
        np.testing.assert_allclose(o2, o1, rtol=1e-4, atol=2e-5)
        np.testing.assert_allclose(l2, l1, rtol=1e-5, atol=2e-5)
    else:
        assert np.abs(o2 - o1).max() <= 2 * BF16_O_ATOL
        assert np.abs(l2 - l1).max() <= 2 * BF16_LSE_ATOL


def test_deterministic_repeat():
    q, k, v = make_qkv(2, 2, 1000, 128, seed=33, dtype="bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = attn_fwd(qd, kd, vd, causal=True)
    o2, l2 = attn_fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_non_default_stream():
    q, k, v = make_qkv(1, 4, 777, 64, seed=34, dtype="bf16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o, lse = attn_fwd(qd, kd, vd, causal=False, stream=s)
    s.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, _scale(64), False)
    assert_close("bf16", o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, 5.0,
                 "stream")
