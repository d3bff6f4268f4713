"""nvfp4_sm_skinny_gb300: small-M skinny GEMM with a deterministic split-K
reduction and its fused epilogues (pre-expert RMSNorm + NVFP4, attention
boundary dual norm) for GB300 (sm_103a).

This module is a thin ctypes binding over ``libsk.so`` (C ABI in
``include/sk.h``). It only marshals torch tensors (device pointers, the current
stream) into the C calls and allocates outputs the caller did not pass; every
step of the computation runs in the library's CUDA kernels. There is no CPU or
PyTorch fallback: if ``libsk.so`` is missing or cannot be loaded, the first
call raises.

Build the library with ``python -c "import __graft_entry__ as g; g.build()"``
or ``python nvfp4_sm_skinny_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsk.so")

SK_OK = 0
SK_ERR_INVALID_ARG = 1
SK_ERR_UNSUPPORTED = 2
SK_ERR_ARCH = 3
SK_ERR_WORKSPACE = 4
SK_ERR_CUDA = 5
SK_ERR_DEVICE_TIMEOUT = 6
MAX_M = 16

_lock = threading.Lock()
_lib = None


class SkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[sk status {status}] {message}")
        self.status = status


class SkValueError(ValueError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[sk status {status}] {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libsk.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libsk.so not found at {LIB_PATH}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "sk_last_error": ([], ctypes.c_char_p),
            "sk_version": ([], i),
            "sk_gemm_splits": ([i, i, i, i], i),
            "sk_gemm_supported": ([i, i, i, i], i),
            "sk_gemm_bf16": ([vp, vp, vp, i, i, i, i, vp], i),
            "sk_gemm_prefetch_next": ([vp, i, i], i),
            "sk_gemm_bf16_ex": ([vp, vp, vp, i, i, i, i, ctypes.c_uint, vp], i),
            "sk_rmsnorm_nvfp4": ([vp, vp, f, f, vp, vp, vp, vp, i, i, vp], i),
            "sk_gemm_rmsnorm_nvfp4_workspace": ([i, i], sz),
            "sk_gemm_rmsnorm_nvfp4": ([vp, vp, vp, f, f, vp, vp, vp, vp, vp, sz, i, i, i, i, vp], i),
            "sk_nvfp4_quantize": ([vp, vp, vp, vp, i, i, vp], i),
            "sk_rmsnorm_bf16": ([vp, vp, f, f, vp, i, i, vp], i),
            "sk_gemm_rmsnorm_bf16": ([vp, vp, vp, f, f, vp, vp, sz, i, i, i, i, vp], i),
            "sk_dual_norm_residual": ([vp, vp, vp, f, vp, vp, vp, f, f, f, f, i, i, vp], i),
            "sk_gemm_dual_norm_workspace": ([i, i], sz),
            "sk_gemm_dual_norm": ([vp, vp, vp, vp, f, vp, vp, vp, f, f, f, f, vp, sz, i, i, i, i, vp], i),
            "sk_gemm_rmsnorm_nvfp4_static": ([vp, vp, vp, f, f, vp, vp, vp, vp, i, i, i, i, vp], i),
            "sk_gemm_nvfp4w_bf16": ([vp, vp, vp, vp, vp, i, i, i, i, vp], i),
            "sk_gemm_nvfp4w_supported": ([i, i, i, i], i),
            "sk_gemm_nvfp4w_splits": ([i, i, i, i], i),
            "sk_device_status": ([ctypes.POINTER(ctypes.c_uint32), i], i),
            "sk_convert_probe": ([i, vp, vp, i, vp], i),
            "sk_wait_probe": ([ctypes.c_uint, vp], i),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def last_error() -> str:
    return lib().sk_last_error().decode()


def _check(status: int) -> None:
    if status == SK_OK:
        return
    msg = last_error()
    if status in (SK_ERR_INVALID_ARG, SK_ERR_UNSUPPORTED, SK_ERR_WORKSPACE):
        raise SkValueError(status, msg)
    raise SkError(status, msg)


def _ptr(t) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, needs {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, needs {tuple(shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: needs a contiguous CUDA tensor")


def version() -> int:
    return int(lib().sk_version())


def gemm_supported(m: int, n: int, k: int, splits: int = 0) -> str | None:
    """None if (m, n, k, splits) has a launch, else the reason."""
    st = lib().sk_gemm_supported(m, n, k, splits)
    return None if st == SK_OK else last_error()


def gemm_splits(m: int, n: int, k: int, splits: int = 0) -> int:
    s = int(lib().sk_gemm_splits(m, n, k, splits))
    if s == 0:
        raise SkValueError(SK_ERR_UNSUPPORTED, last_error())
    return s


# ----------------------------------------------------------------- GEMM ----
GEMM_X_READY = 0x1


def gemm_bf16(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
              splits: int = 0, stream=None, x_ready: bool = False) -> torch.Tensor:
    """out[m, n] = x[m, k] @ w[n, k]^T (BF16 in/out, FP32 accumulate).
    ``x_ready``: no kernel that writes x can still be running when this GEMM
    starts (x written by host copies, or by kernels before a copy, event wait,
    non-overlapped launch or synchronisation), so the GEMM reads it without
    waiting for the kernel ahead of it (sk_gemm_bf16_ex, SK_GEMM_X_READY)."""
    m, k = x.shape
    n = w.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(w, torch.bfloat16, (n, k), "w")
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (m, n), "out")
    if x_ready:
        _check(lib().sk_gemm_bf16_ex(_ptr(x), _ptr(w), _ptr(out), m, n, k, splits, GEMM_X_READY,
                                     _stream(stream)))
    else:
        _check(lib().sk_gemm_bf16(_ptr(x), _ptr(w), _ptr(out), m, n, k, splits, _stream(stream)))
    return out


def gemm_prefetch_next(w_next: torch.Tensor | None) -> None:
    """Hint for the next GEMM this thread enqueues: once it has issued its own
    weight copies, it starts the first weight stages of the GEMM with weight
    ``w_next`` [n, k] (BF16) towards L2. ``None`` clears the hint."""
    if w_next is None:
        _check(lib().sk_gemm_prefetch_next(None, 0, 0))
        return
    _need(w_next, torch.bfloat16, tuple(w_next.shape), "w_next")
    n, k = w_next.shape
    _check(lib().sk_gemm_prefetch_next(_ptr(w_next), n, k))


# -------------------------------------------------------- RMSNorm + NVFP4 ----
def _nvfp4_outputs(m, n, device, a, a_sf):
    if a is None:
        a = torch.empty(m, n // 2, dtype=torch.uint8, device=device)
    if a_sf is None:
        a_sf = torch.empty(m, n // 16, dtype=torch.uint8, device=device)
    _need(a, torch.uint8, (m, n // 2), "a")
    _need(a_sf, torch.uint8, (m, n // 16), "a_sf")
    return a, a_sf


def rmsnorm_nvfp4(y, norm_w, eps: float, gain_center: float, global_scale, a=None, a_sf=None,
                  z_out=None, stream=None):
    """(a, a_sf, z_out): pre-expert RMSNorm of BF16 y [m, n] then NVFP4.
    ``z_out`` may be a tensor, True (allocate) or None (not stored)."""
    m, n = y.shape
    _need(y, torch.bfloat16, (m, n), "y")
    _need(norm_w, torch.bfloat16, (n,), "norm_w")
    _need(global_scale, torch.float32, (1,), "global_scale")
    a, a_sf = _nvfp4_outputs(m, n, y.device, a, a_sf)
    if z_out is True:
        z_out = torch.empty(m, n, dtype=torch.bfloat16, device=y.device)
    if z_out is not None:
        _need(z_out, torch.bfloat16, (m, n), "z_out")
    _check(lib().sk_rmsnorm_nvfp4(_ptr(y), _ptr(norm_w), eps, gain_center, _ptr(global_scale),
                                  _ptr(a), _ptr(a_sf), _ptr(z_out), m, n, _stream(stream)))
    return a, a_sf, z_out


def rmsnorm_bf16(y, norm_w, eps: float, gain_center: float, out=None, stream=None):
    """z BF16 [m, n]: pre-expert RMSNorm of a BF16 edge layer (no NVFP4)."""
    m, n = y.shape
    _need(y, torch.bfloat16, (m, n), "y")
    _need(norm_w, torch.bfloat16, (n,), "norm_w")
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=y.device)
    _need(out, torch.bfloat16, (m, n), "out")
    _check(lib().sk_rmsnorm_bf16(_ptr(y), _ptr(norm_w), eps, gain_center, _ptr(out), m, n,
                                 _stream(stream)))
    return out


def gemm_rmsnorm_bf16(x, w, norm_w, eps: float, gain_center: float, out=None, workspace=None,
                      splits: int = 0, stream=None):
    """(z, workspace): the pooler GEMM then the pre-expert RMSNorm of a BF16
    edge layer. The workspace (uint8) holds the BF16 GEMM output on return."""
    m, k = x.shape
    n = w.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(w, torch.bfloat16, (n, k), "w")
    _need(norm_w, torch.bfloat16, (n,), "norm_w")
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (m, n), "out")
    if workspace is None:
        workspace = torch.empty(gemm_rmsnorm_nvfp4_workspace(m, n), dtype=torch.uint8,
                                device=x.device)
    _check(lib().sk_gemm_rmsnorm_bf16(
        _ptr(x), _ptr(w), _ptr(norm_w), eps, gain_center, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), m, n, k, splits, _stream(stream)))
    return out, workspace


def gemm_rmsnorm_nvfp4_workspace(m: int, n: int) -> int:
    return int(lib().sk_gemm_rmsnorm_nvfp4_workspace(m, n))


def gemm_rmsnorm_nvfp4(x, w, norm_w, eps: float, gain_center: float, global_scale, a=None,
                       a_sf=None, z_out=None, workspace=None, splits: int = 0, stream=None):
    """(a, a_sf, z_out, workspace): the pooler GEMM, pre-expert RMSNorm and
    NVFP4. The workspace (uint8) holds the BF16 GEMM output on return."""
    m, k = x.shape
    n = w.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(w, torch.bfloat16, (n, k), "w")
    _need(norm_w, torch.bfloat16, (n,), "norm_w")
    _need(global_scale, torch.float32, (1,), "global_scale")
    a, a_sf = _nvfp4_outputs(m, n, x.device, a, a_sf)
    if z_out is True:
        z_out = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    if z_out is not None:
        _need(z_out, torch.bfloat16, (m, n), "z_out")
    need = gemm_rmsnorm_nvfp4_workspace(m, n)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check(lib().sk_gemm_rmsnorm_nvfp4(
        _ptr(x), _ptr(w), _ptr(norm_w), eps, gain_center, _ptr(global_scale), _ptr(a), _ptr(a_sf),
        _ptr(z_out), _ptr(workspace), workspace.numel() * workspace.element_size(), m, n, k,
        splits, _stream(stream)))
    return a, a_sf, z_out, workspace


STATIC_SCRATCH_BYTES = 16 * 8192 * 2


def gemm_rmsnorm_nvfp4_static(x, w, norm_w, eps: float, gain_center: float, global_scale, a,
                              a_sf, z_out=None, splits: int = 0, stream=None):
    """The pooler call without a workspace (the library's static device
    scratch holds the GEMM output; m * n <= 131072). The caller passes every
    output; nothing is allocated."""
    m, k = x.shape
    n = w.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(w, torch.bfloat16, (n, k), "w")
    _need(norm_w, torch.bfloat16, (n,), "norm_w")
    _need(global_scale, torch.float32, (1,), "global_scale")
    _need(a, torch.uint8, (m, n // 2), "a")
    _need(a_sf, torch.uint8, (m, n // 16), "a_sf")
    if z_out is not None:
        _need(z_out, torch.bfloat16, (m, n), "z_out")
    _check(lib().sk_gemm_rmsnorm_nvfp4_static(
        _ptr(x), _ptr(w), _ptr(norm_w), eps, gain_center, _ptr(global_scale), _ptr(a), _ptr(a_sf),
        _ptr(z_out), m, n, k, splits, _stream(stream)))
    return a, a_sf, z_out


def nvfp4_quantize(z, global_scale, a=None, a_sf=None, stream=None):
    """(a, a_sf): NVFP4 of BF16 z [m, n]."""
    m, n = z.shape
    _need(z, torch.bfloat16, (m, n), "z")
    _need(global_scale, torch.float32, (1,), "global_scale")
    a, a_sf = _nvfp4_outputs(m, n, z.device, a, a_sf)
    _check(lib().sk_nvfp4_quantize(_ptr(z), _ptr(global_scale), _ptr(a), _ptr(a_sf), m, n,
                                   _stream(stream)))
    return a, a_sf


# ------------------------------------------------------------- dual norm ----
def dual_norm_residual(partial, resid, post_w, alpha: float, beta, pre_w, out=None,
                       eps_post: float = 1e-6, eps_pre: float = 1e-6, gc_post: float = 0.0,
                       gc_pre: float = 0.0, stream=None):
    """out: post_attn_norm(partial), gated add into resid (FP32, in place),
    pre_ffn_norm into BF16 out."""
    m, h = partial.shape
    _need(partial, torch.bfloat16, (m, h), "partial")
    _need(resid, torch.float32, (m, h), "resid")
    if post_w is not None:
        _need(post_w, torch.bfloat16, (h,), "post_w")
    _need(beta, torch.bfloat16, (h,), "beta")
    _need(pre_w, torch.bfloat16, (h,), "pre_w")
    if out is None:
        out = torch.empty(m, h, dtype=torch.bfloat16, device=partial.device)
    _need(out, torch.bfloat16, (m, h), "out")
    _check(lib().sk_dual_norm_residual(_ptr(partial), _ptr(resid), _ptr(post_w), alpha, _ptr(beta),
                                       _ptr(pre_w), _ptr(out), eps_post, eps_pre, gc_post, gc_pre,
                                       m, h, _stream(stream)))
    return out


def gemm_dual_norm_workspace(m: int, n: int) -> int:
    return int(lib().sk_gemm_dual_norm_workspace(m, n))


def gemm_dual_norm(x, w, resid, post_w, alpha: float, beta, pre_w, out=None,
                   eps_post: float = 1e-6, eps_pre: float = 1e-6, gc_post: float = 0.0,
                   gc_pre: float = 0.0, workspace=None, splits: int = 0, stream=None):
    """(out, workspace): o_proj GEMM then the dual norm. The workspace holds the
    BF16 partial on return."""
    m, k = x.shape
    n = w.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(w, torch.bfloat16, (n, k), "w")
    _need(resid, torch.float32, (m, n), "resid")
    if post_w is not None:
        _need(post_w, torch.bfloat16, (n,), "post_w")
    _need(beta, torch.bfloat16, (n,), "beta")
    _need(pre_w, torch.bfloat16, (n,), "pre_w")
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (m, n), "out")
    need = gemm_dual_norm_workspace(m, n)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check(lib().sk_gemm_dual_norm(
        _ptr(x), _ptr(w), _ptr(resid), _ptr(post_w), alpha, _ptr(beta), _ptr(pre_w), _ptr(out),
        eps_post, eps_pre, gc_post, gc_pre, _ptr(workspace),
        workspace.numel() * workspace.element_size(), m, n, k, splits, _stream(stream)))
    return out, workspace


# ------------------------------------------------- weight-only NVFP4 GEMM ----
def gemm_nvfp4w_supported(m: int, n: int, k: int, splits: int = 0) -> str | None:
    """None if the weight-only NVFP4 GEMM has a launch for the shape, else why."""
    st = lib().sk_gemm_nvfp4w_supported(m, n, k, splits)
    return None if st == SK_OK else last_error()


def gemm_nvfp4w_splits(m: int, n: int, k: int, splits: int = 0) -> int:
    s = int(lib().sk_gemm_nvfp4w_splits(m, n, k, splits))
    if s == 0:
        raise SkValueError(SK_ERR_UNSUPPORTED, last_error())
    return s


def gemm_nvfp4w(x, wq, wsf, w_scale, out=None, splits: int = 0, stream=None):
    """out[m, n] = bf16(w_scale * x[m, k] @ W^T), W[n, k] = e2m1(wq) * e4m3(wsf):
    wq uint8 [n, k/2] (column 2c in the low nibble), wsf uint8 [n, k/16]
    (float8_e4m3fn bits), w_scale float32 [1] on the device."""
    m, k = x.shape
    n = wq.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(wq, torch.uint8, (n, k // 2), "wq")
    _need(wsf, torch.uint8, (n, k // 16), "wsf")
    _need(w_scale, torch.float32, (1,), "w_scale")
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (m, n), "out")
    _check(lib().sk_gemm_nvfp4w_bf16(_ptr(x), _ptr(wq), _ptr(wsf), _ptr(w_scale), _ptr(out), m, n,
                                     k, splits, _stream(stream)))
    return out


# ----------------------------------------------------------- diagnostics ----
def device_status(clear: bool = True) -> int:
    """The device status word (OR of SK_DEVICE_WAIT_* bits); synchronizes."""
    v = ctypes.c_uint32(0)
    _check(lib().sk_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


SK_DEVICE_WAIT_PROBE = 0x10


def wait_probe(limit_us: int, stream=None) -> None:
    """Launches a kernel whose bounded wait is meant to run out after limit_us
    microseconds; it sets SK_DEVICE_WAIT_PROBE in the device status word."""
    _check(lib().sk_wait_probe(limit_us, _stream(stream)))


def convert_probe(kind: int, inp: torch.Tensor, stream=None) -> torch.Tensor:
    """Runs one device format conversion over ``inp`` (see sk_convert_probe)."""
    n = inp.numel()
    if kind == 3:
        _need(inp, torch.uint8, (n,), "inp")
        out = torch.empty(n, dtype=torch.float32, device=inp.device)
    else:
        _need(inp, torch.float32, (n,), "inp")
        out = torch.empty(n, dtype=torch.int16 if kind == 2 else torch.uint8, device=inp.device)
    _check(lib().sk_convert_probe(kind, _ptr(inp), _ptr(out), n, _stream(stream)))
    return out
