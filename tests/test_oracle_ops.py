"""Pins for the oracle's GEMM, pre-expert RMSNorm, NVFP4 quantizer and dual norm.

Each check is tied to something other than the oracle's own formula: the
hand-worked fixtures in tests/golden (cited to the page passages), exact
rational arithmetic, closed forms and invariants (identity and one-hot
weights, scale invariance, special cases of the dual norm), and numpy's FP64
matmul as a library routine.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_cases

f32 = np.float32


def bf16_bits(vals) -> np.ndarray:
    """Bits of values that are exactly representable in BF16 (checked)."""
    a = np.asarray(vals, np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture value not exact in BF16"
    return (u >> 16).astype(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def trunc_bf16(vals) -> np.ndarray:
    """Bits of the BF16 value obtained by truncating each FP32 value."""
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rand_bf16(rng, shape, std=1.0, mean=0.0):
    return trunc_bf16(rng.standard_normal(shape) * std + mean)


def exact_bf16_round(v: Fraction) -> int:
    """BF16 bits nearest to the exact rational v, ties to even, -0 -> +0."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = math.floor(math.log2(float(a)))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    lo = (a // q)
    rem = a - lo * q
    if rem * 2 > q or (rem * 2 == q and lo % 2 == 1):
        lo += 1
    val = float(lo * q)
    return int(np.array([val], np.float32).view(np.uint32)[0] >> 16) | sign


# ------------------------------------------------------------------ GEMM ----
def test_gemm_golden(oracle_mod):
    for case in read_cases("gemm_worked.txt"):
        m, n, k = int(case["m"][0]), int(case["n"][0]), int(case["k"][0])
        x = bf16_bits([float(v) for v in case["x"]]).reshape(m, k)
        w = bf16_bits([float(v) for v in case["w"]]).reshape(n, k)
        want = np.array([int(h, 16) for h in case["y_bits"]], np.uint16).reshape(m, n)
        assert np.array_equal(oracle_mod.gemm_bf16(x, w), want), case


def test_gemm_identity(oracle_mod):
    rng = np.random.default_rng(0)
    for k in (16, 64, 256):
        x = rand_bf16(rng, (3, k))
        w = bf16_bits(np.eye(k, dtype=np.float32))
        y = oracle_mod.gemm_bf16(x, w)
        want = np.where(x == 0x8000, 0, x)          # -0 is stored as +0
        assert np.array_equal(y, want)


def test_gemm_one_hot_power_of_two(oracle_mod):
    rng = np.random.default_rng(1)
    m, n, k = 5, 48, 96
    x = bits_to_f64(rand_bf16(rng, (m, k))).astype(np.float32)
    x = np.clip(x, -1e30, 1e30)
    perm = rng.integers(0, k, n)
    cs = 2.0 ** rng.integers(-4, 5, n)
    w = np.zeros((n, k), np.float32)
    w[np.arange(n), perm] = cs
    y = bits_to_f64(oracle_mod.gemm_bf16(bf16_bits(x), bf16_bits(w)))
    assert np.array_equal(y, x[:, perm].astype(np.float64) * cs[None, :])


def test_gemm_exact_rational_small(oracle_mod):
    # Brute force with exact rationals on tiny integer-and-dyadic inputs; the
    # oracle must equal the correctly rounded exact sum.
    rng = np.random.default_rng(2)
    for trial in range(30):
        m, n, k = rng.integers(1, 5), rng.integers(1, 9), rng.integers(1, 40)
        xv = (rng.integers(-64, 65, (m, k)) / 8.0).astype(np.float32)
        wv = (rng.integers(-128, 129, (n, k)) / 32.0).astype(np.float32)
        y = oracle_mod.gemm_bf16(bf16_bits(xv), bf16_bits(wv))
        for i in range(m):
            for j in range(n):
                s = sum(Fraction(float(xv[i, t])) * Fraction(float(wv[j, t])) for t in range(k))
                assert y[i, j] == exact_bf16_round(s)


def test_gemm_m1_dot_products_correctly_rounded(oracle_mod):
    # Random BF16 dot products (K up to 4096): the oracle equals the exactly
    # rounded rational sum unless that sum lies within the FP64 summation error
    # of a BF16 midpoint (then either neighbour is acceptable).
    rng = np.random.default_rng(3)
    for k in (1, 7, 64, 1024, 4096):
        x = rand_bf16(rng, (1, k))
        w = rand_bf16(rng, (16, k), std=0.02)
        y = oracle_mod.gemm_bf16(x, w)
        xf, wf = bits_to_f64(x), bits_to_f64(w)
        for j in range(16):
            prods = [Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[0], wf[j])]
            s = sum(prods)
            want = exact_bf16_round(s)
            if y[0, j] != want:
                bound = k * 2.0 ** -53 * float(sum(abs(p) for p in prods))
                lo = bits_to_f64(np.array([want], np.uint16))[0]
                assert abs(float(s) - lo) > 0 and bound > 0
                # must be a near-midpoint case
                ulp = 2.0 ** (math.floor(math.log2(abs(lo))) - 7)
                assert abs(abs(float(s) - lo) - ulp / 2) <= bound


def test_gemm_zero_input_gives_positive_zero(oracle_mod):
    rng = np.random.default_rng(4)
    w = rand_bf16(rng, (32, 64))
    y = oracle_mod.gemm_bf16(np.zeros((4, 64), np.uint16), w)
    assert np.all(y == 0)
    # negative-zero inputs too: (-0) * w sums to a zero whose sign varies
    y = oracle_mod.gemm_bf16(np.full((2, 64), 0x8000, np.uint16), w)
    assert np.all(y == 0)


def test_gemm_f64_matches_numpy(oracle_mod):
    rng = np.random.default_rng(5)
    x, w = rand_bf16(rng, (7, 300)), rand_bf16(rng, (33, 300), 0.02)
    acc, absacc = oracle_mod.gemm_f64(x, w)
    xf, wf = bits_to_f64(x), bits_to_f64(w)
    ref = xf @ wf.T
    np.testing.assert_allclose(acc, ref, rtol=0, atol=1e-12 * (np.abs(xf) @ np.abs(wf).T).max())
    np.testing.assert_allclose(absacc, np.abs(xf) @ np.abs(wf).T, rtol=1e-13)


# --------------------------------------------------------------- RMSNorm ----
def test_rmsnorm_golden(oracle_mod):
    for case in read_cases("rmsnorm_worked.txt"):
        m, n = int(case["m"][0]), int(case["n"][0])
        y = bf16_bits([float(v) for v in case["y"]]).reshape(m, n)
        w = bf16_bits([float(v) for v in case["w"]])
        z = oracle_mod.rmsnorm_bf16(y, w, float(case["eps"][0]), float(case["gain_center"][0]))
        want = np.array([int(h, 16) for h in case["z_bits"]], np.uint16).reshape(m, n)
        assert np.array_equal(z, want)


def test_rmsnorm_unit_rows(oracle_mod):
    # With eps = 0 and weight + gain_center = 1, every element of a row with
    # constant magnitude normalises to +-1 exactly.
    rng = np.random.default_rng(6)
    n = 256
    for c in (0.001, 1.0, 3.0, 1000.0):
        signs = rng.choice([-1.0, 1.0], n).astype(np.float32)
        y = trunc_bf16(signs * np.float32(c))
        w = bf16_bits(np.full(n, 0.0, np.float32))
        z = oracle_mod.rmsnorm_bf16(y[None], w, 0.0, 1.0)
        assert np.array_equal(bits_to_f64(z[0]), signs.astype(np.float64))


def test_rmsnorm_constant_row_closed_form(oracle_mod):
    n = 4096
    for c, g, eps in ((0.5, 1.0, 1e-6), (2.0, 1.25, 1e-6), (0.0009765625, 1.0, 1e-6)):
        y = bf16_bits(np.full(n, c, np.float32))
        w = bf16_bits(np.full(n, g - 1.0, np.float32))
        z = oracle_mod.rmsnorm_bf16(y[None], w, eps, 1.0)
        e = float(np.float32(eps))
        want = exact_bf16_round(Fraction(c / math.sqrt(c * c + e) * g))
        assert np.all(z == want)


def test_rmsnorm_scale_invariance_and_zero_row(oracle_mod):
    rng = np.random.default_rng(7)
    y = rand_bf16(rng, (3, 512))
    w = rand_bf16(rng, (512,), 0.1)
    z1 = oracle_mod.rmsnorm_bf16(y, w, 0.0, 1.0)
    y2 = bf16_bits(bits_to_f64(y).astype(np.float32) * 4)   # exact scaling
    z2 = oracle_mod.rmsnorm_bf16(y2, w, 0.0, 1.0)
    assert np.array_equal(z1, z2)
    z0 = oracle_mod.rmsnorm_bf16(np.zeros((1, 512), np.uint16), w, 1e-6, 1.0)
    assert np.all(z0 == 0)


def test_rmsnorm_weight_after_norm(oracle_mod):
    # pooler_layer: the weight multiplies the normalised value (it does not
    # enter the mean). Doubling w + gain_center doubles z exactly (eps = 0),
    # while the mean is unchanged.
    rng = np.random.default_rng(8)
    y = rand_bf16(rng, (2, 64))
    w = bf16_bits(np.full(64, 0.25, np.float32))          # w + 1 = 1.25
    w2 = bf16_bits(np.full(64, 1.5, np.float32))          # w + 1 = 2.5
    z1 = bits_to_f64(oracle_mod.rmsnorm_bf16(y, w, 0.0, 1.0))
    z2 = bits_to_f64(oracle_mod.rmsnorm_bf16(y, w2, 0.0, 1.0))
    assert np.array_equal(z1 * 2, z2)


# ----------------------------------------------------------------- NVFP4 ----
def test_nvfp4_golden(oracle_mod):
    for case in read_cases("nvfp4_worked.txt"):
        z = bf16_bits([float(v) for v in case["z"]])[None]
        a, a_sf = oracle_mod.nvfp4_quantize(z, float(case["gs"][0]))
        assert a_sf[0, 0] == int(case["sf"][0], 16), case
        assert [int(v) for v in a[0]] == [int(h, 16) for h in case["a"]], case


def test_nvfp4_exactly_representable_roundtrip(oracle_mod):
    # gs = 1 and a power-of-two scale 2^e exact in e4m3: if every block holds
    # one 6 * 2^e and other values in the e2m1 grid times 2^e, then
    # sf = 2^e and every code is recovered exactly.
    rng = np.random.default_rng(9)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)
    for e in (-6, -2, 0, 3, 6):
        codes = rng.integers(0, 16, (4, 64))
        codes[:, ::16] = 7
        vals = grid[codes & 7] * np.where(codes & 8, -1, 1) * np.float32(2.0 ** e)
        vals[vals == 0] = 0.0                                  # +0 as stored
        codes = np.where((codes & 7) == 0, 0, codes)
        a, a_sf = oracle_mod.nvfp4_quantize(bf16_bits(vals), 1.0)
        assert np.all(a_sf == oracle_mod.e4m3_from_float(2.0 ** e))
        unpacked = np.stack([a & 0xF, a >> 4], -1).reshape(4, 64)
        assert np.array_equal(unpacked, codes)


def test_nvfp4_zero_blocks_give_zero_scale_and_codes(oracle_mod):
    # an all-zero block: amax = 0, sf = 0x00, os = 0 and every code 0x0 (z is
    # canonical +0); a zero block next to a non-zero one is unaffected by it
    z = np.zeros((3, 64), np.float32)
    z[1, 16:32] = 1.5
    a, a_sf = oracle_mod.nvfp4_quantize(bf16_bits(z), 100.0)
    assert np.all(a_sf[0] == 0) and np.all(a[0] == 0) and np.all(a[2] == 0)
    assert a_sf[1, 0] == 0 and a_sf[1, 2] == 0 and a_sf[1, 3] == 0 and a_sf[1, 1] != 0
    assert np.all(a[1, :8] == 0) and np.all(a[1, 16:] == 0) and np.all(a[1, 8:16] == 0x77)


def test_nvfp4_constant_row_same_code_every_block(oracle_mod):
    z = bf16_bits(np.full((2, 256), -1.375, np.float32))
    a, a_sf = oracle_mod.nvfp4_quantize(z, 37.0)
    assert np.all(a_sf == a_sf[0, 0]) and np.all(a == a[0, 0])
    assert (a[0, 0] & 0xF) == (a[0, 0] >> 4) == 0xF        # amax maps to 6


def test_nvfp4_codes_are_nearest_after_scaling(oracle_mod):
    # Brute-force check of every code on random blocks: the chosen e2m1 value
    # is the grid point nearest |z * os| (FP32 product), ties to even code.
    rng = np.random.default_rng(10)
    z = rand_bf16(rng, (8, 512))
    gs = 2688.0 / 4.0
    a, a_sf = oracle_mod.nvfp4_quantize(z, gs)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    zf = bits_to_f64(z).astype(np.float32)
    codes = np.stack([a & 0xF, a >> 4], -1).reshape(8, 512)
    for i in range(8):
        for b in range(32):
            blk = zf[i, 16 * b:16 * b + 16]
            amax = np.max(np.abs(blk))
            sf = oracle_mod.e4m3_from_float(float(f32(f32(amax / f32(6.0)) * f32(gs))))
            assert a_sf[i, b] == sf
            sff = f32(oracle_mod.e4m3_to_float(sf))
            os_ = f32(0.0) if sff == 0 else f32(1.0) / (sff * (f32(1.0) / f32(gs)))
            for j in range(16):
                v = Fraction(float(f32(blk[j] * os_)))
                mag = min(range(8), key=lambda c: (abs(Fraction(grid[c]) - abs(v)), c & 1))
                if abs(v) > 6:
                    mag = 7
                assert codes[i, 16 * b + j] & 7 == mag
                assert bool(codes[i, 16 * b + j] & 8) == (blk[j] < 0 or (blk[j] == 0 and np.signbit(blk[j])))


def test_nvfp4_saturates_beyond_calibration(oracle_mod):
    z = bf16_bits(np.array([100.0] + [1.0] * 15, np.float32))[None]
    a, a_sf = oracle_mod.nvfp4_quantize(z, 2688.0 / 10.0)   # amax 100 > calibrated 10
    assert a_sf[0, 0] == 0x7E and (a[0, 0] & 0xF) == 7


# ------------------------------------------------------------- dual norm ----
def _dual_case(case):
    h = int(case["h"][0])
    p = bf16_bits([float(v) for v in case["p"]])[None]
    s = np.array([[float(v) for v in case["s"]]], np.float32)
    w1 = None if case["w1"] == ["none"] else bf16_bits([float(v) for v in case["w1"]])
    beta = bf16_bits([float(v) for v in case["beta"]])
    w2 = bf16_bits([float(v) for v in case["w2"]])
    return h, p, s, w1, beta, w2


def test_dual_norm_golden(oracle_mod):
    for case in read_cases("dual_norm_worked.txt"):
        h, p, s, w1, beta, w2 = _dual_case(case)
        eps = float(case["eps"][0])
        s2, out = oracle_mod.dual_norm(p, s, w1, float(case["alpha"][0]), beta, w2, eps, eps,
                                       float(case["gc_post"][0]), float(case["gc_pre"][0]))
        assert np.array_equal(s2[0], np.array([float(v) for v in case["s_out"]], np.float32))
        assert [int(v) for v in out[0]] == [int(hx, 16) for hx in case["out_bits"]]


def _rand_dual(rng, m=3, h=1024):
    p = rand_bf16(rng, (m, h))
    s = rng.standard_normal((m, h)).astype(np.float32)
    w1 = rand_bf16(rng, (h,), 0.1, mean=1.0)
    beta = rand_bf16(rng, (h,), 1.0)
    w2 = rand_bf16(rng, (h,), 0.5)
    return p, s, w1, beta, w2


def test_dual_norm_beta_zero_leaves_stream_and_norms_it(oracle_mod):
    rng = np.random.default_rng(11)
    p, s, w1, _, w2 = _rand_dual(rng)
    beta0 = np.zeros(w2.shape, np.uint16)
    s2, out = oracle_mod.dual_norm(p, s, w1, 1.0, beta0, w2, 1e-6, 1e-6)
    assert np.array_equal(s2, s)
    # out = RMSNorm(s) * w2: for rows of s that are exact BF16 values this is
    # the oracle's pre-expert RMSNorm with gain_center 0 (an independent path).
    sb = bf16_bits(bits_to_f64(rand_bf16(rng, s.shape)).astype(np.float32))
    sf = bits_to_f64(sb).astype(np.float32)
    s3, out3 = oracle_mod.dual_norm(p, sf, w1, 1.0, beta0, w2, 1e-6, 1e-6)
    assert np.array_equal(out3, oracle_mod.rmsnorm_bf16(sb, w2, 1e-6, 0.0))


def test_dual_norm_alpha_zero_is_gated_post_norm(oracle_mod):
    # alpha = 0: s' = float(beta * q); with beta = 1 and no post weight,
    # s' is the post-norm of p, i.e. the pre-expert RMSNorm of p with unit
    # weight, before BF16 rounding -- compare after rounding.
    rng = np.random.default_rng(12)
    p, s, _, _, w2 = _rand_dual(rng)
    ones = bf16_bits(np.ones(w2.shape, np.float32))
    s2, _ = oracle_mod.dual_norm(p, s, None, 0.0, ones, w2, 1e-6, 1e-6)
    zeros_w = np.zeros(w2.shape, np.uint16)
    z = oracle_mod.rmsnorm_bf16(p, zeros_w, 1e-6, 1.0)
    # BF16 rounding of the FP32 stream equals the BF16 RMSNorm except where
    # the FP32 rounding moved a value across a BF16 midpoint (double rounding)
    sb = np.array([[oracle_mod.bf16_from_double(float(v)) for v in row] for row in s2], np.uint16)
    sb = np.where(sb == 0x8000, 0, sb)
    assert np.mean(sb != z) < 1e-3


def test_dual_norm_null_post_weight_equals_unit_weight(oracle_mod):
    rng = np.random.default_rng(13)
    p, s, _, beta, w2 = _rand_dual(rng)
    ones = bf16_bits(np.ones(w2.shape, np.float32))
    a = oracle_mod.dual_norm(p, s, None, 0.75, beta, w2, 1e-6, 1e-6)
    b = oracle_mod.dual_norm(p, s, ones, 0.75, beta, w2, 1e-6, 1e-6, gc_post=0.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_dual_norm_gain_center_shifts_weight(oracle_mod):
    # (w + gc) with w = 0.5, gc = 0.5 must equal w = 1.0, gc = 0
    rng = np.random.default_rng(14)
    p, s, _, beta, _ = _rand_dual(rng)
    h = p.shape[1]
    half = bf16_bits(np.full(h, 0.5, np.float32))
    one = bf16_bits(np.full(h, 1.0, np.float32))
    a = oracle_mod.dual_norm(p, s, half, 1.0, beta, half, 1e-6, 1e-6, 0.5, 0.5)
    b = oracle_mod.dual_norm(p, s, one, 1.0, beta, one, 1e-6, 1e-6, 0.0, 0.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_dual_norm_stream_update_matches_fp64_numpy(oracle_mod):
    # the gated residual, s' = fl32(alpha*s + beta*q), against numpy FP64 with
    # q from the library's own sum of squares
    rng = np.random.default_rng(15)
    p, s, w1, beta, w2 = _rand_dual(rng)
    s2, _ = oracle_mod.dual_norm(p, s, w1, 0.9, beta, w2, 1e-6, 1e-6)
    pf = bits_to_f64(p)
    r1 = 1 / np.sqrt(np.mean(pf * pf, axis=1, keepdims=True) + float(f32(1e-6)))
    q = pf * r1 * bits_to_f64(w1)[None]
    want = (float(f32(0.9)) * s.astype(np.float64) + bits_to_f64(beta)[None] * q)
    np.testing.assert_allclose(s2, want.astype(np.float32), rtol=2e-7, atol=1e-30)
