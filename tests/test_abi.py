"""Host-side tests of the C ABI: the library builds, loads without a GPU, exports
every function include/sk.h declares, and rejects invalid arguments before any
CUDA call (the validation mirrors the unpooler page's launch_unsupported)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def sk():
    from nvfp4_sm_skinny_gb300 import build

    build.build()
    import nvfp4_sm_skinny_gb300 as sk

    return sk


def header_functions():
    src = open(os.path.join(ROOT, "include", "sk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sk_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for want in ("sk_gemm_bf16", "sk_gemm_rmsnorm_nvfp4", "sk_rmsnorm_nvfp4", "sk_nvfp4_quantize",
                 "sk_dual_norm_residual", "sk_gemm_dual_norm", "sk_last_error", "sk_version"):
        assert want in names


def test_library_exports_every_header_symbol(sk):
    lib = ctypes.CDLL(sk.LIB_PATH)
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert sk.version() == 1


# Fake, 16-byte-aligned device addresses: validation must reject the shape
# before anything dereferences them or touches CUDA.
P = 1 << 20


@pytest.mark.parametrize("m,n,k,splits,status", [
    (0, 128, 64, 0, 1), (17, 128, 64, 0, 1),          # m outside 1..16
    (1, 0, 64, 0, 1), (1, 24, 64, 0, 1),               # n not a positive multiple of 16
    (1, 128, 0, 0, 1), (1, 128, 96, 0, 1),             # k not a multiple of 64
    (1, 128, 64, 3, 2), (1, 128, 64, 32, 2),           # split count not in the set
    (1, 128, 192, 2, 2),                               # K does not split evenly
])
def test_gemm_shape_validation(sk, m, n, k, splits, status):
    lib = sk.lib()
    assert lib.sk_gemm_supported(m, n, k, splits) == status
    assert sk.last_error()
    st = lib.sk_gemm_bf16(ctypes.c_void_p(P), ctypes.c_void_p(P), ctypes.c_void_p(P), m, n, k,
                          splits, None)
    assert st == status


def test_gemm_supported_ok(sk):
    lib = sk.lib()
    for args in ((1, 1024, 4096, 0), (16, 8192, 4096, 2), (16, 16, 64, 1), (5, 4096, 8192, 16)):
        assert lib.sk_gemm_supported(*args) == 0
    assert sk.gemm_supported(16, 8192, 1024, 4) is None
    assert "split" in sk.gemm_supported(16, 8192, 1024, 3)


def test_pointer_validation(sk):
    lib = sk.lib()
    vp = ctypes.c_void_p
    assert lib.sk_gemm_bf16(None, vp(P), vp(P), 1, 128, 64, 0, None) == 1
    assert "null" in sk.last_error()
    assert lib.sk_gemm_bf16(vp(P + 8), vp(P), vp(P), 1, 128, 64, 0, None) == 1
    assert "aligned" in sk.last_error()
    # workspace too small
    st = lib.sk_gemm_rmsnorm_nvfp4(vp(P), vp(P), vp(P), 1e-6, 1.0, vp(P), vp(P), vp(P), None,
                                   vp(P), 16, 4, 4096, 8192, 0, None)
    assert st == 4 and "workspace" in sk.last_error()
    assert lib.sk_gemm_rmsnorm_nvfp4_workspace(16, 4096) == 16 * 4096 * 2
    assert lib.sk_gemm_dual_norm_workspace(3, 8192) == (3 * 8192 * 2 + 255) // 256 * 256


def test_prefetch_hint_validation(sk):
    # the hint is host state only: it is checked and stored without CUDA
    lib = sk.lib()
    vp = ctypes.c_void_p
    assert lib.sk_gemm_prefetch_next(None, 0, 0) == 0          # clears
    assert lib.sk_gemm_prefetch_next(vp(P), 24, 64) == 1        # n not a multiple of 16
    assert lib.sk_gemm_prefetch_next(vp(P), 128, 96) == 1       # k not a multiple of 64
    assert lib.sk_gemm_prefetch_next(vp(P + 8), 128, 64) == 1
    assert "aligned" in sk.last_error()
    assert lib.sk_gemm_prefetch_next(vp(P), 128, 64) == 0
    assert lib.sk_gemm_prefetch_next(None, 0, 0) == 0


def test_gemm_ex_validation(sk):
    lib = sk.lib()
    vp = ctypes.c_void_p
    assert lib.sk_gemm_bf16_ex(vp(P), vp(P), vp(P), 1, 128, 64, 0, 2, None) == 1   # unknown flag
    assert "flags" in sk.last_error()
    assert lib.sk_gemm_bf16_ex(vp(P), vp(P), vp(P), 1, 24, 64, 0, 1, None) == 1    # bad n
    assert lib.sk_gemm_bf16_ex(vp(P + 8), vp(P), vp(P), 1, 128, 64, 0, 1, None) == 1


def test_epilogue_validation(sk):
    lib = sk.lib()
    vp = ctypes.c_void_p
    # rmsnorm/nvfp4: n not a multiple of 16, m too big
    assert lib.sk_rmsnorm_nvfp4(vp(P), vp(P), 1e-6, 1.0, vp(P), vp(P), vp(P), None, 1, 40,
                                None) == 1
    assert lib.sk_rmsnorm_nvfp4(vp(P), vp(P), 1e-6, 1.0, vp(P), vp(P), vp(P), None, 17, 64,
                                None) == 1
    # global scale misaligned
    assert lib.sk_nvfp4_quantize(vp(P), vp(P + 2), vp(P), vp(P), 1, 64, None) == 1
    # dual norm: h too large / not a multiple of 8
    assert lib.sk_dual_norm_residual(vp(P), vp(P), None, 1.0, vp(P), vp(P), vp(P), 1e-6, 1e-6,
                                     0.0, 0.0, 1, 8200, None) == 1
    assert lib.sk_dual_norm_residual(vp(P), vp(P), None, 1.0, vp(P), vp(P), vp(P), 1e-6, 1e-6,
                                     0.0, 0.0, 1, 12, None) == 1
    assert lib.sk_convert_probe(9, vp(P), vp(P), 4, None) == 1


def test_valid_call_without_gpu_reports_device_error(sk):
    # On a machine without a GB300 a well-formed call fails cleanly with a
    # device error (no usable device or wrong architecture), never a crash.
    import torch

    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    lib = sk.lib()
    vp = ctypes.c_void_p
    st = lib.sk_gemm_bf16(vp(P), vp(P), vp(P), 1, 128, 64, 0, None)
    assert st in (3, 5) and sk.last_error()


def test_binding_raises_value_error_on_bad_tensors(sk):
    import torch

    x = torch.zeros(2, 64, dtype=torch.float32)
    w = torch.zeros(128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sk.gemm_bf16(x, w)


@pytest.mark.parametrize("m,n,k,splits,status", [
    (0, 128, 256, 0, 1), (17, 128, 256, 0, 1),        # m outside 1..16
    (1, 24, 256, 0, 1),                                 # n not a multiple of 16
    (1, 128, 128, 0, 1), (1, 128, 320, 0, 1),           # k not a multiple of 256
    (1, 128, 256, 3, 2), (1, 128, 512, 4, 2),           # split count / uneven split
])
def test_nvfp4w_shape_validation(sk, m, n, k, splits, status):
    lib = sk.lib()
    vp = ctypes.c_void_p
    assert lib.sk_gemm_nvfp4w_supported(m, n, k, splits) == status
    assert sk.last_error()
    st = lib.sk_gemm_nvfp4w_bf16(vp(P), vp(P), vp(P), vp(P), vp(P), m, n, k, splits, None)
    assert st == status


def test_nvfp4w_pointer_validation(sk):
    lib = sk.lib()
    vp = ctypes.c_void_p
    assert lib.sk_gemm_nvfp4w_supported(16, 8192, 8192, 0) == 0
    assert lib.sk_gemm_nvfp4w_bf16(vp(P), None, vp(P), vp(P), vp(P), 1, 128, 256, 0, None) == 1
    assert lib.sk_gemm_nvfp4w_bf16(vp(P), vp(P), vp(P + 8), vp(P), vp(P), 1, 128, 256, 0, None) == 1
    assert "aligned" in sk.last_error()
    assert lib.sk_gemm_nvfp4w_bf16(vp(P), vp(P), vp(P), vp(P + 2), vp(P), 1, 128, 256, 0, None) == 1
    assert "w_scale" in sk.last_error()
