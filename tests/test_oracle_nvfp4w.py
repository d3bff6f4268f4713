"""Pins of the oracle's weight-only NVFP4 GEMM (oracle_gemm_nvfp4w,
oracle_nvfp4_dequant). Not on the pages: the weight W [n, k] is held in the
NVFP4 byte layout of the pooler page's module docstring (cutedsl/moe/
pooler_gather: two e2m1 codes per byte with column 2c in the low nibble, one
float8_e4m3fn scale per 16 columns of a row) and one FP32 multiplier w_scale;
y = bf16_rn(w_scale * sum_k x W). Each pin is independent of the oracle's own
arithmetic: hand-worked fixtures, torch's float8_e4m3fn decoding and the
e2m1 value table, the already pinned BF16 GEMM and NVFP4 quantizer, and
closed-form scalings."""
import numpy as np
import pytest
import torch

from conftest import read_cases

# e2m1 magnitudes of codes 0..7 (bit 3 is the sign), as the pooler page's
# cvt_e2m1x8_f32 helper decodes them
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def bf16_bits(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def e4m3_values(b):
    """float8_e4m3fn bytes -> float64 through torch's own decoding."""
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def independent_dequant(wq, wsf):
    """W [n, k] from the bytes, decoded here with the table above and torch."""
    n = wq.shape[0]
    codes = np.stack([wq & 0xF, wq >> 4], -1).reshape(n, -1)        # even column low
    vals = E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    return vals * np.repeat(e4m3_values(wsf), 16, axis=1)


def random_weight(rng, n, k):
    wq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    wsf = rng.integers(0, 0x7F, (n, k // 16), dtype=np.uint8)     # finite scales
    return wq, wsf


def test_gemm_nvfp4w_golden(oracle_mod):
    for case in read_cases("gemm_nvfp4w_worked.txt"):
        m, n, k = int(case["m"][0]), int(case["n"][0]), int(case["k"][0])
        x = bf16_bits([float(v) for v in case["x"]]).reshape(m, k)
        wq = np.array([int(h, 16) for h in case["wq"]], np.uint8).reshape(n, k // 2)
        wsf = np.array([int(h, 16) for h in case["wsf"]], np.uint8).reshape(n, k // 16)
        want = np.array([int(h, 16) for h in case["y_bits"]], np.uint16).reshape(m, n)
        got = oracle_mod.gemm_nvfp4w(x, wq, wsf, float(case["w_scale"][0]))
        assert np.array_equal(got, want), (case, got)


def test_dequant_matches_independent_decode(oracle_mod):
    rng = np.random.default_rng(1)
    wq, wsf = random_weight(rng, 7, 96)
    assert np.array_equal(oracle_mod.nvfp4_dequant(wq, wsf), independent_dequant(wq, wsf))


def test_one_hot_rows_pick_single_weights(oracle_mod):
    # x row i is the unit vector at column j_i: y[i, r] = bf16(w_scale * W[r, j_i]).
    # Columns cover even and odd positions and both sides of a block boundary.
    rng = np.random.default_rng(2)
    n, k = 12, 64
    wq, wsf = random_weight(rng, n, k)
    cols = [0, 1, 14, 15, 16, 17, 31, 32, 47, 62, 63]
    x = np.zeros((len(cols), k), np.float32)
    x[np.arange(len(cols)), cols] = 1.0
    W = independent_dequant(wq, wsf)
    for w_scale in (1.0, 0.125):
        got = oracle_mod.gemm_nvfp4w(bf16_bits(x), wq, wsf, w_scale)
        want = bf16_bits(w_scale * W[:, cols].T)       # exact: <= 6 significant bits
        want = np.where(want == 0x8000, 0, want)
        assert np.array_equal(got, want), w_scale


@pytest.mark.parametrize("e,g", [(0, 0), (-3, 2), (2, -4), (-6, 5)])
def test_quantized_representable_weight_equals_bf16_gemm(oracle_mod, e, g):
    # W with one 6 * 2^e per block and every value on the e2m1 grid times 2^e;
    # quantized by the (already pinned) NVFP4 quantizer with gs = 2^g gives
    # scale 2^(e+g) and the exact codes, so w_scale = 2^-g restores W exactly
    # and the weight-only GEMM must equal the BF16 GEMM of W bit for bit.
    rng = np.random.default_rng(100 + 31 * (e + 10) + (g + 10))
    n, k, m = 9, 128, 5
    codes = rng.integers(0, 16, (n, k))
    codes[:, ::16] = 7
    W = (E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0) * 2.0 ** e).astype(np.float32)
    Wb = bf16_bits(W)
    Wb = np.where(Wb == 0x8000, 0, Wb)
    wq, wsf = oracle_mod.nvfp4_quantize(Wb, 2.0 ** g)
    assert np.all(e4m3_values(wsf) == 2.0 ** (e + g))
    assert np.array_equal(oracle_mod.nvfp4_dequant(wq, wsf) * 2.0 ** -g, W.astype(np.float64))
    x = bf16_bits(rng.standard_normal((m, k)))
    y = oracle_mod.gemm_nvfp4w(x, wq, wsf, 2.0 ** -g)
    assert np.array_equal(y, oracle_mod.gemm_bf16(x, Wb))


def test_sum_matches_float64_matmul(oracle_mod):
    rng = np.random.default_rng(4)
    m, n, k = 3, 10, 256
    wq, wsf = random_weight(rng, n, k)
    x = bf16_bits(rng.standard_normal((m, k)))
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    W = independent_dequant(wq, wsf)
    y, acc, absacc = oracle_mod.gemm_nvfp4w(x, wq, wsf, 0.75, return_acc=True)
    ref = 0.75 * (xf @ W.T)
    assert np.all(np.abs(acc - ref) <= 1e-14 * (0.75 * np.abs(xf) @ np.abs(W).T) + 1e-300)
    assert np.allclose(absacc, 0.75 * (np.abs(xf) @ np.abs(W).T), rtol=1e-14)
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert np.all(np.abs(yf - ref) <= 0.5 * ulp * (1 + 1e-12))   # one rounding


def test_w_scale_scales_exactly(oracle_mod):
    # acc is linear in w_scale: a power of two scales it exactly (w_scale
    # multiplies the sum; dividing by it would fail this)
    rng = np.random.default_rng(5)
    wq, wsf = random_weight(rng, 6, 64)
    x = bf16_bits(rng.standard_normal((2, 64)))
    _, a1, _ = oracle_mod.gemm_nvfp4w(x, wq, wsf, 1.0, return_acc=True)
    for p in (-5, -1, 3):
        _, ap, _ = oracle_mod.gemm_nvfp4w(x, wq, wsf, 2.0 ** p, return_acc=True)
        assert np.array_equal(ap, a1 * 2.0 ** p)


def test_zero_scales_and_zero_w_scale(oracle_mod):
    rng = np.random.default_rng(6)
    n, k = 5, 64
    wq, wsf = random_weight(rng, n, k)
    x = bf16_bits(rng.standard_normal((3, k)))
    # a block with scale 0 contributes nothing, whatever its codes
    wsf0 = wsf.copy()
    wsf0[:, 2] = 0
    wq0 = wq.copy()
    wq0[:, 16:24] = 0
    assert np.array_equal(oracle_mod.gemm_nvfp4w(x, wq, wsf0, 1.0),
                          oracle_mod.gemm_nvfp4w(x, wq0, wsf0, 1.0))
    # w_scale 0 (either sign) gives +0.0 everywhere
    for ws in (0.0, -0.0):
        assert np.all(oracle_mod.gemm_nvfp4w(x, wq, wsf, ws) == 0)
