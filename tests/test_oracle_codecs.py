"""Pins for the oracle's number-format codecs (BF16, float8_e4m3fn, e2m1).

Each codec is checked against something other than itself: torch's own
float32 -> bfloat16 / float8_e4m3fn casts (library routines, round to nearest
even), exact rational arithmetic (fractions.Fraction) and brute-force nearest
search over the whole value grid.
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_cases

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf16_bits_torch(vals_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(vals_f32.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _nearest_bf16_exact(v: Fraction) -> int:
    """Brute force: BF16 bits of the representable value nearest to v (ties to
    even last bit), by comparing exact distances to the neighbours found from
    FP32 candidates."""
    if v == 0:
        return 0
    # candidates: all BF16 values around float(v)
    f = float(v)
    u = int(np.array([f], np.float32).view(np.uint32)[0]) >> 16
    best = None
    for b in range(max(0, (u & 0x7FFF) - 2), min(0x7F80, (u & 0x7FFF) + 3)):
        for s in (0, 0x8000):
            bits = b | s
            val = Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))
            d = abs(val - v)
            key = (d, bits & 1)
            if best is None or key < best[0]:
                best = (key, bits)
    return best[1]


def test_bf16_roundtrip_all_patterns(oracle_mod):
    for b in range(1 << 16):
        e = (b >> 7) & 0xFF
        m = b & 0x7F
        if e == 0xFF and m != 0:
            continue  # NaN encodings
        v = oracle_mod.bf16_to_double(b)
        assert oracle_mod.bf16_from_double(v) == b, hex(b)


def test_bf16_matches_torch_on_float32_inputs(oracle_mod):
    rng = np.random.default_rng(7)
    # every BF16 value, the exact midpoints between neighbours, and one FP32
    # ulp to either side of each midpoint
    base = (np.arange(0, 0x7F7F, dtype=np.uint32) << 16)
    mids = base | 0x8000
    vals = np.concatenate([base, mids, mids + 1, mids - 1]).view(np.float32)
    vals = np.concatenate([vals, -vals, rng.standard_normal(20000).astype(np.float32) * 100])
    vals = vals[np.isfinite(vals)]
    sample = vals[rng.choice(len(vals), 60000, replace=False)]
    want = _bf16_bits_torch(sample)
    got = np.array([oracle_mod.bf16_from_double(float(v)) for v in sample], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounds_straight_from_double(oracle_mod):
    # A double just above a BF16 midpoint whose FP32 rounding lands exactly on
    # the midpoint: rounding through FP32 would tie to even (down); rounding
    # straight from FP64 must go up. Checked against exact brute force.
    rng = random.Random(3)
    for _ in range(400):
        b = rng.randrange(0x0080, 0x7F00)
        lo = Fraction(float(np.array([b << 16], np.uint32).view(np.float32)[0]))
        hi = Fraction(float(np.array([(b + 1) << 16], np.uint32).view(np.float32)[0]))
        mid = (lo + hi) / 2
        for delta in (Fraction(1, 1 << 40), -Fraction(1, 1 << 40), Fraction(0)):
            v = mid + delta * mid
            want = _nearest_bf16_exact(v)
            assert oracle_mod.bf16_from_double(float(v)) == want
            assert oracle_mod.bf16_from_double(-float(v)) == want | 0x8000


def test_bf16_sign_and_limits(oracle_mod):
    assert oracle_mod.bf16_from_double(-0.0) == 0x8000
    assert oracle_mod.bf16_from_double(0.0) == 0
    assert oracle_mod.bf16_from_double(3.3895313892515355e38) == 0x7F7F  # max finite
    assert oracle_mod.bf16_from_double(3.5e38) == 0x7F80                 # overflow -> inf
    assert oracle_mod.bf16_from_double(2.0 ** -133) == 0x0001           # smallest subnormal
    assert oracle_mod.bf16_from_double(2.0 ** -134) == 0x0000           # tie -> even (0)
    assert oracle_mod.bf16_from_double(3 * 2.0 ** -135) == 0x0001


def test_e4m3_decode_all_bytes_matches_torch(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for b in range(256):
        got = oracle_mod.e4m3_to_float(b)
        if math.isnan(ref[b]):
            assert math.isnan(got)
        else:
            assert got == ref[b] and math.copysign(1, got) == math.copysign(1, ref[b]), b


def test_e4m3_encode_matches_torch_in_range(oracle_mod):
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = np.unique(np.abs(vals[np.isfinite(vals)]))
    mids = (finite[1:] + finite[:-1]) / 2
    probe = np.concatenate([finite, mids]).astype(np.float32)
    probe = np.concatenate([probe, np.nextafter(probe, np.float32(0)),
                            np.nextafter(probe, np.float32(np.inf))])
    probe = probe[np.abs(probe) <= 448]
    rng = np.random.default_rng(11)
    probe = np.concatenate([probe, (rng.random(20000) * 448).astype(np.float32),
                            np.exp2(rng.uniform(-12, 8.8, 20000)).astype(np.float32)])
    probe = probe[probe <= 448]
    probe = np.concatenate([probe, -probe])
    want = torch.from_numpy(probe).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_from_float(float(v)) for v in probe], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(probe[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_e4m3_roundtrip_and_saturation(oracle_mod):
    for b in range(256):
        if (b & 0x7F) == 0x7F:
            continue
        assert oracle_mod.e4m3_from_float(oracle_mod.e4m3_to_float(b)) == b
    # .satfinite: finite overflow clamps to the largest finite magnitude
    assert oracle_mod.e4m3_from_float(448.0) == 0x7E
    assert oracle_mod.e4m3_from_float(464.0) == 0x7E     # tie 448 | (480 = NaN slot)
    assert oracle_mod.e4m3_from_float(470.0) == 0x7E
    assert oracle_mod.e4m3_from_float(1e30) == 0x7E
    assert oracle_mod.e4m3_from_float(-1e30) == 0xFE
    assert oracle_mod.e4m3_from_float(2.0 ** -9) == 0x01  # smallest subnormal
    assert oracle_mod.e4m3_from_float(2.0 ** -10) == 0x00  # tie -> even (0)
    assert oracle_mod.e4m3_from_float(3 * 2.0 ** -11) == 0x01  # 0.75 of a step -> 1
    assert oracle_mod.e4m3_from_float(5 * 2.0 ** -11) == 0x01  # 1.25 steps -> 1
    assert oracle_mod.e4m3_from_float(3 * 2.0 ** -10) == 0x02  # 1.5 steps: tie -> even 2


def _e2m1_brute(v: float) -> int:
    """Nearest e2m1 magnitude by exhaustive search, ties to the even code,
    finite overflow clamped to 6; sign in bit 3."""
    a = abs(Fraction(v))
    best = min(range(8), key=lambda c: (abs(Fraction(E2M1_GRID[c]) - a), c & 1))
    if a > 6:
        best = 7
    return best | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_brute_force_grid(oracle_mod):
    grid = [c * 0.03125 for c in range(-320, 321)]          # [-10, 10] step 1/32
    mids = [(a + b) / 2 for a, b in zip(E2M1_GRID, E2M1_GRID[1:])]
    extra = []
    for m in mids:
        f = np.float32(m)
        extra += [float(f), float(np.nextafter(f, np.float32(0))), float(np.nextafter(f, np.float32(9)))]
    rng = np.random.default_rng(5)
    extra += list(rng.uniform(-8, 8, 5000).astype(np.float32).astype(float))
    for v in grid + extra + [-x for x in extra]:
        assert oracle_mod.e2m1_from_float(v) == _e2m1_brute(v), v


def test_e2m1_decode(oracle_mod):
    for c in range(16):
        mag = E2M1_GRID[c & 7]
        got = oracle_mod.e2m1_to_float(c)
        assert abs(got) == mag and (math.copysign(1, got) < 0) == bool(c & 8)


def test_e2m1_ties_and_saturation_fixture(oracle_mod):
    # ties -> even code; > 6 saturates (cvt_e2m1x8_f32 is round-to-nearest,
    # saturating); fixture values come from the nvfp4 worked example at gs = 1
    case = read_cases("nvfp4_worked.txt")[0]
    z = [float(v) for v in case["z"]]
    codes = [oracle_mod.e2m1_from_float(v) for v in z]
    packed = [codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(8)]
    assert packed == [int(h, 16) for h in case["a"]]
    assert oracle_mod.e2m1_from_float(7.0) == 7 and oracle_mod.e2m1_from_float(1e9) == 7
    assert oracle_mod.e2m1_from_float(-7.0) == 0xF


@pytest.mark.parametrize("v", [-0.2, -0.25, -1e-30])
def test_e2m1_negative_underflow_keeps_sign(oracle_mod, v):
    # Reading of the pages' silence: the sign survives rounding to zero, as in
    # IEEE rounding; the device cvt parity test checks the hardware agrees.
    assert oracle_mod.e2m1_from_float(v) == 0x8
