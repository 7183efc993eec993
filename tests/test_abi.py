"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects invalid arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from attention_attn_fwd_05_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "attn_fwd.h")


@pytest.fixture(scope="module")
def L():
    from attention_attn_fwd_05_gb300.build import build
    build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert set(declared_functions()) == set(binding.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings_and_version(L):
    for code in range(13):
        assert L.attn_status_string(code) != b"unknown status", code
    assert L.attn_status_string(999) == b"unknown status"
    assert L.attn_version() == 10200


# Fake, never-dereferenced addresses: validation must reject these calls
# before any CUDA call is made.
A = 0x7F0000001000


def call(L, q=A, k=A, v=A, o=A + 0x100000, lse=None, B=1, H=1, N=128, d=64, dtype=1,
         scale=0.125):
    return L.attn_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), 0, dtype, None)


BAD_SCALES = [float("nan"), float("inf"), float("-inf"), 3.0e38, -3.0e38]


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("scale", BAD_SCALES)
def test_non_finite_scale_rejected(L, dtype, scale):
    """The softmax multiplier must be finite (|scale| <= 2e38): ATTN_ERR_SCALE
    from every entry point that takes one, before any CUDA call."""
    f = ctypes.c_float(scale)
    assert call(L, dtype=dtype, scale=scale) == 11
    assert L.attn_fwd_noalloc(A, A, A, A + 0x100000, None, 1, 1, 128, 64, f, 0, dtype,
                              None) == 11
    ws = L.attn_fwd_host_workspace_bytes(1, 1, 128, 64, dtype)
    assert L.attn_fwd_host(A, A, A, A + 0x100000, None, 1, 1, 128, 64, f, 1, dtype,
                           A + 0x200000, ws, None) == 11
    assert L.attn_bwd(*([A] * 10), 1, 1, 128, 64, f, 0, dtype, None) == 11


def test_shape_errors_come_before_the_scale_check(L):
    assert call(L, N=0, scale=float("nan")) == 2
    assert call(L, d=96, scale=float("nan")) == 4


def test_null_pointers_rejected(L):
    assert call(L, q=None) == 1
    assert call(L, k=None) == 1
    assert call(L, v=None) == 1
    assert call(L, o=None) == 1


@pytest.mark.parametrize("B,H,N", [(0, 1, 1), (1, 0, 1), (1, 1, 0), (-1, 1, 1), (1, 1, 2 ** 31),
                                   (2 ** 30, 2 ** 30, 2 ** 10)])
def test_bad_shapes_rejected(L, B, H, N):
    assert call(L, B=B, H=H, N=N) == 2


def test_bf16_sequence_limit(L):
    assert call(L, N=65535 * 128 + 1) == 2


def test_bf16_grid_limit(L):
    """B*H*ceil(N/256) items must fit the kernels' 1-D grid (< 2^31)."""
    assert call(L, B=1024, H=128, N=65535 * 128) == 2
    assert call(L, B=1024, H=128, N=65535 * 128, dtype=0) == 2  # and fp32: B*H > 65535


def test_f32_head_limit(L):
    assert call(L, B=65536, H=1, N=1, dtype=0) == 2


@pytest.mark.parametrize("dtype", [-1, 2, 7])
def test_bad_dtype_rejected(L, dtype):
    assert call(L, dtype=dtype) == 3


@pytest.mark.parametrize("d", [0, 32, 96, 256, 63])
def test_bad_head_dim_rejected(L, d):
    assert call(L, d=d) == 4


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_misaligned_rejected(L, which):
    kw = {which: A + 8}
    assert call(L, **kw) == 5


def test_row_softmax_validation(L):
    assert L.attn_row_softmax(None, A, None, 1, 1, None) == 1
    assert L.attn_row_softmax(A, A, None, 0, 1, None) == 2
    assert L.attn_row_softmax(A, A, None, 1, 0, None) == 2
    assert L.attn_row_softmax(A + 2, A, None, 1, 4, None) == 5


def test_python_wrapper_value_errors():
    import torch
    from attention_attn_fwd_05_gb300 import attn_fwd, row_softmax
    x = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        attn_fwd(x, x, x)  # CPU tensors
    with pytest.raises(ValueError):
        row_softmax(torch.zeros(3, 4))


def test_add_rmsnorm_validation(L):
    f = ctypes.c_float(1e-6)
    assert L.attn_add_rmsnorm(None, None, A, A, None, 1, 8, f, 0, None) == 1
    assert L.attn_add_rmsnorm(A, A, A, A, None, 1, 8, f, 0, None) == 1   # residual needs res_out
    assert L.attn_add_rmsnorm(A, None, A, A, None, 0, 8, f, 0, None) == 2
    assert L.attn_add_rmsnorm(A, None, A, A, None, 1, 0, f, 0, None) == 2
    assert L.attn_add_rmsnorm(A, None, A, A, None, 1, 2 ** 31, f, 0, None) == 2
    assert L.attn_add_rmsnorm(A, None, A, A, None, 1, 8, f, 5, None) == 3
    assert L.attn_add_rmsnorm(A + 4, None, A, A, None, 1, 8, f, 0, None) == 5


def test_attn_bwd_validation(L):
    f = ctypes.c_float(0.125)
    args = [A] * 10
    assert L.attn_bwd(None, *args[1:], 1, 1, 8, 64, f, 0, 1, None) == 1
    assert L.attn_bwd(*args, 0, 1, 8, 64, f, 0, 1, None) == 2
    assert L.attn_bwd(*args, 1, 1, 8, 64, f, 0, 9, None) == 3
    assert L.attn_bwd(*args, 1, 1, 8, 96, f, 0, 1, None) == 4
    assert L.attn_bwd(*args, 65536, 1, 8, 64, f, 0, 1, None) == 2
    bad = list(args)
    bad[6] = A + 4
    assert L.attn_bwd(*bad, 1, 1, 8, 64, f, 0, 1, None) == 5


def test_fwd_host_rejects_bad_arguments_on_the_host(L):
    """attn_fwd_host validates before touching CUDA: NULL pointers, shapes,
    a workspace that is too small or misaligned."""
    ws_need = L.attn_fwd_host_workspace_bytes(1, 2, 300, 64, 1)
    # Q, K, V, O at 2 B per element and LSE at 4 B, each rounded up to 256 B.
    assert ws_need == 4 * 76800 + 2560
    assert L.attn_fwd_host_workspace_bytes(1, 2, 300, 65, 1) == 0
    assert L.attn_fwd_host_workspace_bytes(0, 2, 300, 64, 1) == 0
    assert L.attn_fwd_host_workspace_bytes(1, 2, 300, 64, 7) == 0

    def host(q=A, k=A, v=A, o=A + 0x100000, ws=A + 0x200000, nbytes=ws_need, N=300, d=64,
             dtype=1):
        return L.attn_fwd_host(q, k, v, o, None, 1, 2, N, d, ctypes.c_float(0.125), 1, dtype,
                               ws, nbytes, None)
    assert host(q=None) == 1
    assert host(o=None) == 1
    assert host(ws=None) == 1
    assert host(d=96) == 4
    assert host(dtype=5) == 3
    assert host(nbytes=ws_need - 1) == 2
    assert host(ws=A + 0x200080) == 5


def test_noalloc_objects_reference_no_device_allocator(L):
    """The object files on attn_fwd_noalloc's path (the entry point itself and
    the two kernel launchers it calls) reference no CUDA allocation or free
    routine.  attn_api.o, which holds attn_fwd's per-device set-up, does: the
    check can tell them apart.  (A static check of our own build's symbol
    tables; the GPU test in test_zz_no_alloc.py checks the device's free
    memory.)"""
    import subprocess
    from attention_attn_fwd_05_gb300.build import BUILD
    pat = re.compile(r"^(cuda|cu)(Malloc|Free|MemAlloc|MemFree|HostAlloc|MemPool|"
                     r"MallocAsync|FreeAsync|MallocManaged|MallocPitch|Malloc3D|MallocArray)")

    def alloc_refs(obj):
        out = subprocess.run(["nm", "-u", os.path.join(BUILD, obj)], capture_output=True,
                             text=True, check=True).stdout
        return [ln.split()[-1] for ln in out.splitlines() if pat.match(ln.split()[-1])]

    for obj in ("attn_noalloc.o", "attn_fwd_tc.o", "attn_fwd_f32.o"):
        assert alloc_refs(obj) == [], obj
    assert "cudaMalloc" in alloc_refs("attn_api.o")
