"""CPU oracle: a plain, slow, single-threaded C statement of the hot path.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this package. The product library (the CUDA path) never
does, and the two share no code: this wrapper only marshals numpy arrays into
``oracle.c`` through ctypes.

Conventions: BF16 tensors are numpy ``uint16`` arrays of raw bits, e4m3 and
packed e2m1 are ``uint8``, the FP32 residual stream is ``float32``.

Functions and the page passages they follow (vLLM API pages of the Muse Spark
specialized decode):

* ``gemm_bf16`` / ``gemm_f64``: cutedsl/gemm/unpooler, module docstring (the
  small-M product) and cutedsl/moe/pooler_gather, compile_pooler_gemm.
* ``rmsnorm_bf16``: cutedsl/moe/pooler_gather, module docstring (the pre-expert
  norm) and pooler_layer (weight applied after the norm).
* ``nvfp4_quantize``: cutedsl/moe/pooler_gather, module docstring (NVFP4 layout),
  cvt_e2m1x8_f32, cvt_f32_to_e4m3, nvfp4_compute_output_scale.
* ``dual_norm``: cutedsl/oproj/batt, AttentionBoundary.
* ``nvfp4_dequant`` / ``gemm_nvfp4w``: not on the pages. The weight-only
  NVFP4 GEMM holds W [n, k] in the NVFP4 layout of the pooler page's module
  docstring (codes two per byte, even column low nibble; one e4m3 scale per
  16 columns of a row) with one FP32 multiplier ``w_scale``.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, library routines (torch's float8/bfloat16 casts),
brute force and hand-worked fixtures in ``tests/golden``. Nothing is
"parity unpinned" except what the design notes list.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fno-fast-math"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, no threads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        i = ctypes.c_int
        d = ctypes.c_double
        vp = ctypes.c_void_p

        lib.oracle_bf16_from_double.argtypes = [d]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = d
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_e4m3_to_float.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_float.restype = ctypes.c_float
        lib.oracle_e2m1_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_from_float.restype = ctypes.c_uint8
        lib.oracle_e2m1_to_float.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_to_float.restype = ctypes.c_float
        lib.oracle_gemm_f64.argtypes = [u16p, u16p, vp, vp, i, i, i]
        lib.oracle_gemm_f64.restype = None
        lib.oracle_gemm_bf16.argtypes = [u16p, u16p, u16p, i, i, i]
        lib.oracle_gemm_bf16.restype = None
        lib.oracle_rmsnorm_bf16.argtypes = [u16p, u16p, d, d, u16p, vp, i, i]
        lib.oracle_rmsnorm_bf16.restype = None
        lib.oracle_nvfp4_quantize.argtypes = [u16p, ctypes.c_float, u8p, u8p, i, i]
        lib.oracle_nvfp4_quantize.restype = None
        lib.oracle_dual_norm.argtypes = [u16p, f32p, vp, d, u16p, u16p, u16p,
                                         d, d, d, d, vp, vp, i, i]
        lib.oracle_dual_norm.restype = None
        lib.oracle_nvfp4_dequant.argtypes = [u8p, u8p, f64p, i, i]
        lib.oracle_nvfp4_dequant.restype = None
        lib.oracle_gemm_nvfp4w.argtypes = [u16p, u8p, u8p, ctypes.c_float, vp, vp, vp, i, i, i]
        lib.oracle_gemm_nvfp4w.restype = None
        _lib = lib
        return lib


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def _f32(v: float) -> float:
    # Scalars cross the product's C ABI as FP32; the oracle takes the same value.
    return float(np.float32(v))


def _ptr(a) -> ctypes.c_void_p | None:
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- codecs ----
def bf16_from_double(v: float) -> int:
    """BF16 bits of ``v`` rounded to nearest, ties to even, straight from FP64."""
    return int(_load().oracle_bf16_from_double(float(v)))


def bf16_to_double(b: int) -> float:
    return float(_load().oracle_bf16_to_double(int(b)))


def e4m3_from_float(v: float) -> int:
    """float8_e4m3fn bits of the FP32 value ``v``: round to nearest even, finite
    overflow saturated to +-448."""
    return int(_load().oracle_e4m3_from_float(float(np.float32(v))))


def e4m3_to_float(b: int) -> float:
    return float(_load().oracle_e4m3_to_float(int(b)))


def e2m1_from_float(v: float) -> int:
    """e2m1 code (sign in bit 3) of the FP32 value ``v``: round to nearest,
    ties to the even code, overflow saturated to +-6."""
    return int(_load().oracle_e2m1_from_float(float(np.float32(v))))


def e2m1_to_float(c: int) -> float:
    return float(_load().oracle_e2m1_to_float(int(c)))


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode BF16 bit patterns (uint16) into float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ GEMM ----
def gemm_f64(x, w):
    """(acc, absacc): the FP64 k-ordered sums x @ w^T and sum |x*w|, [m, n]."""
    x, w = _u16(x), _u16(w)
    m, k = x.shape
    n = w.shape[0]
    assert w.shape[1] == k
    acc = np.empty((m, n), np.float64)
    absacc = np.empty((m, n), np.float64)
    _load().oracle_gemm_f64(x, w, _ptr(acc), _ptr(absacc), m, n, k)
    return acc, absacc


def gemm_bf16(x, w) -> np.ndarray:
    """y[m, n] = bf16_rn(sum_k x[m,k] w[n,k]) with -0 stored as +0 (uint16 bits)."""
    x, w = _u16(x), _u16(w)
    m, k = x.shape
    n = w.shape[0]
    assert w.shape[1] == k
    y = np.empty((m, n), np.uint16)
    _load().oracle_gemm_bf16(x, w, y, m, n, k)
    return y


# --------------------------------------------------------------- RMSNorm ----
def rmsnorm_bf16(y, w, eps: float, gain_center: float, return_rinv: bool = False):
    """z = bf16(y * rsqrt(mean(y^2) + eps) * (w + gain_center)), row-wise."""
    y, w = _u16(y), _u16(w)
    m, n = y.shape
    assert w.shape == (n,)
    z = np.empty((m, n), np.uint16)
    rinv = np.empty((m,), np.float64)
    _load().oracle_rmsnorm_bf16(y, w, _f32(eps), _f32(gain_center), z, _ptr(rinv), m, n)
    return (z, rinv) if return_rinv else z


# ----------------------------------------------------------------- NVFP4 ----
def nvfp4_quantize(z, global_scale: float):
    """(a [m, n/2] uint8, a_sf [m, n/16] uint8 e4m3fn bits) of BF16 z [m, n]."""
    z = _u16(z)
    m, n = z.shape
    assert n % 16 == 0
    a = np.empty((m, n // 2), np.uint8)
    a_sf = np.empty((m, n // 16), np.uint8)
    _load().oracle_nvfp4_quantize(z, float(np.float32(global_scale)), a, a_sf, m, n)
    return a, a_sf


def rmsnorm_nvfp4(y, w, eps: float, gain_center: float, global_scale: float):
    """(a, a_sf, z): the pre-expert norm of BF16 y, then its NVFP4 quantization."""
    z = rmsnorm_bf16(y, w, eps, gain_center)
    a, a_sf = nvfp4_quantize(z, global_scale)
    return a, a_sf, z


def gemm_rmsnorm_nvfp4(x, w, norm_w, eps: float, gain_center: float, global_scale: float):
    """(a, a_sf, z, y): GEMM, then the pre-expert norm, then NVFP4."""
    y = gemm_bf16(x, w)
    a, a_sf, z = rmsnorm_nvfp4(y, norm_w, eps, gain_center, global_scale)
    return a, a_sf, z, y


# ------------------------------------------------------------- dual norm ----
def dual_norm(partial, stream, post_w, alpha: float, beta, pre_w, eps_post: float,
              eps_pre: float, gc_post: float = 0.0, gc_pre: float = 0.0,
              return_r: bool = False):
    """(stream', out): post_attn_norm of the BF16 partial, gated add into a copy
    of the FP32 stream, pre_ffn_norm of the result into BF16. ``post_w`` may be
    None (no post-norm weight)."""
    p = _u16(partial)
    m, h = p.shape
    s = np.array(stream, dtype=np.float32, copy=True, order="C")
    assert s.shape == (m, h)
    w1 = None if post_w is None else _u16(post_w)
    beta, w2 = _u16(beta), _u16(pre_w)
    out = np.empty((m, h), np.uint16)
    r1 = np.empty((m,), np.float64)
    r2 = np.empty((m,), np.float64)
    _load().oracle_dual_norm(p, s, _ptr(w1), _f32(alpha), beta, w2, out,
                             _f32(eps_post), _f32(eps_pre), _f32(gc_post),
                             _f32(gc_pre), _ptr(r1), _ptr(r2), m, h)
    return (s, out, r1, r2) if return_r else (s, out)


# ------------------------------------------------- weight-only NVFP4 GEMM ----
def nvfp4_dequant(wq, wsf) -> np.ndarray:
    """dq [n, k] float64: e2m1(code) * e4m3(block scale) of NVFP4 weight bytes
    wq [n, k/2] (column 2c in the low nibble) and wsf [n, k/16] (exact)."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
    n, kh = wq.shape
    k = 2 * kh
    assert k % 16 == 0 and wsf.shape == (n, k // 16)
    dq = np.empty((n, k), np.float64)
    _load().oracle_nvfp4_dequant(wq, wsf, dq, n, k)
    return dq


def gemm_nvfp4w(x, wq, wsf, w_scale: float, return_acc: bool = False):
    """y [m, n] BF16 bits = bf16_rn(w_scale * sum_k x[m,k] dq[n,k]), -0 stored as
    +0; with ``return_acc`` also (acc, absacc): w_scale * sum and
    |w_scale| * sum |x dq| in float64."""
    x = _u16(x)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
    m, k = x.shape
    n = wq.shape[0]
    assert wq.shape == (n, k // 2) and wsf.shape == (n, k // 16) and k % 16 == 0
    y = np.empty((m, n), np.uint16)
    acc = np.empty((m, n), np.float64)
    absacc = np.empty((m, n), np.float64)
    _load().oracle_gemm_nvfp4w(x, wq, wsf, _f32(w_scale), _ptr(y), _ptr(acc), _ptr(absacc), m, n, k)
    return (y, acc, absacc) if return_acc else y
