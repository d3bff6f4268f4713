"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (stated here and in the design notes):

* BF16 GEMM output: an element passes if (i) its BF16 value is within one
  unit in the last place of the oracle's correctly rounded FP64 result
  (ordered-bits distance <= 1), or (ii) it lies within
  ulp(gpu)/2 + gamma * sum_k |x w| of the exact FP64 sum, with
  gamma = (K / (16 * S) + 16 + S) * 2^-22: a worst-case bound for FP32
  accumulation of K/(16 S) sequential tensor-core steps of 16 products each,
  plus the S-term split sum. (ii) only matters where the exact result is
  tiny next to the summands (cancellation); the fraction of elements that
  need it must stay below 2e-4 (the worst case seen on GB300 is 6.9e-5).
* BF16 norm outputs computed from the same input: ordered-bits distance <= 1
  (FP32 on the GPU against FP64 in the oracle, one rounding each).
* FP32 residual: |gpu - ref| <= 1e-5 * (|alpha s| + |beta q|) per element.
* NVFP4 from the same BF16 z: bit-exact scales and codes. End to end from x:
  codes at most one step off on at most 1e-3 of the elements, scales at most
  one step off on at most 1e-3 of the blocks, and exact wherever the 16 BF16
  inputs of a block agree bit for bit.
"""
from __future__ import annotations

import math

import numpy as np


def ordinal_bf16(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b).astype(np.int64) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordinal_bf16(a) - ordinal_bf16(b))


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -126)))
    e = np.maximum(e, -126)
    return 2.0 ** (e - 7)


def gemm_gamma(k: int, splits: int) -> float:
    return (k / (16.0 * splits) + 16 + splits) * 2.0 ** -22


# (label, outputs beyond one ulp of the correctly rounded result, outputs,
# largest ulp distance) of every labelled check_gemm call in this session; the
# test session prints them as a table (tests/conftest.py).
GEMM_RECORDS: list = []


def check_gemm(y_gpu_bits, y_ref_bits, acc, absacc, k: int, splits: int, max_frac_ii: float = 2e-4,
               label: str | None = None, gamma_extra: float = 0.0):
    """Asserts the GEMM tolerance; returns (n_strict_fail, n_total, max_ulp).
    n_strict_fail counts the outputs more than one BF16 ulp from the oracle's
    correctly rounded result, i.e. those accepted only by the cancellation
    clause (ii); with a ``label`` the counts are recorded for the session's
    report. ``gamma_extra`` widens gamma for roundings after the sum (the
    weight-only NVFP4 GEMM multiplies the FP32 sum by w_scale: 2^-24)."""
    y_gpu_bits = np.asarray(y_gpu_bits, np.uint16)
    d = ulp_distance(y_gpu_bits, y_ref_bits)
    strict = d <= 1
    g = bf16_to_f64(y_gpu_bits)
    bound = 0.5 * bf16_ulp(g) + (gemm_gamma(k, splits) + gamma_extra) * absacc
    loose = np.abs(g - acc) <= bound
    bad = ~(strict | loose)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), float(g[tuple(i)]), float(acc[tuple(i)]), float(bound[tuple(i)]))
                  for i in idx]
        raise AssertionError(f"{bad.sum()} GEMM outputs outside tolerance: {detail}")
    n_ii = int((~strict).sum())
    if label is not None:
        GEMM_RECORDS.append((label, n_ii, int(d.size), int(d.max())))
    assert n_ii <= max(1, math.ceil(max_frac_ii * d.size)), \
        f"{n_ii} of {d.size} outputs needed the cancellation bound"
    assert not np.any(y_gpu_bits == 0x8000), "negative zero stored"
    return n_ii, d.size, int(d.max())


def e2m1_ordinal(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64)
    mag = c & 7
    return np.where(c & 8, -mag, mag)


def unpack_codes(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, np.uint8)
    return np.stack([a & 0xF, a >> 4], -1).reshape(a.shape[0], -1)


def check_nvfp4_end_to_end(a_gpu, sf_gpu, z_gpu, a_ref, sf_ref, z_ref, frac: float = 1e-3):
    """End-to-end NVFP4 tolerance; returns (n_code_diff, n_sf_diff)."""
    cg, cr = unpack_codes(a_gpu), unpack_codes(a_ref)
    dc = np.abs(e2m1_ordinal(cg) - e2m1_ordinal(cr))
    assert dc.max() <= 1, f"code off by {dc.max()} steps"
    n_code = int((dc != 0).sum())
    assert n_code <= max(1, frac * dc.size), f"{n_code} of {dc.size} codes differ"
    sfg = np.asarray(sf_gpu).astype(np.int64) & 0x7F
    sfr = np.asarray(sf_ref).astype(np.int64) & 0x7F
    ds = np.abs(sfg - sfr)
    assert ds.max() <= 1, f"scale off by {ds.max()} steps"
    n_sf = int((ds != 0).sum())
    assert n_sf <= max(1, frac * ds.size), f"{n_sf} of {ds.size} scales differ"
    # exact wherever the block's BF16 inputs agree
    m, n = np.asarray(z_gpu).shape
    same = (np.asarray(z_gpu).reshape(m, n // 16, 16) == np.asarray(z_ref).reshape(m, n // 16, 16)).all(-1)
    assert np.array_equal(np.asarray(sf_gpu)[same], np.asarray(sf_ref)[same])
    cb_g = cg.reshape(m, n // 16, 16)[same]
    cb_r = cr.reshape(m, n // 16, 16)[same]
    assert np.array_equal(cb_g, cb_r)
    return n_code, n_sf
