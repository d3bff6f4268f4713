"""The device's format conversions used by the NVFP4 epilogue, checked against
the oracle's codecs over every BF16 value (as FP32), dense grids through every
rounding midpoint, and +-0. This pins both sides: the oracle's reading of the
e2m1 / e4m3 rounding (including the sign of a negative value that rounds to
zero) and the hardware's behaviour."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    import nvfp4_sm_skinny_gb300 as sk

    sk.lib()
    return sk


def all_bf16_as_f32():
    b = np.arange(1 << 16, dtype=np.uint32)
    e = (b >> 7) & 0xFF
    keep = e != 0xFF                      # drop inf/NaN
    return (b[keep] << 16).view(np.float32)


def e2m1_probe_inputs():
    grid = np.arange(-8.5, 8.5, 1 / 1024, dtype=np.float64).astype(np.float32)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    mids = (mags[1:] + mags[:-1]) / 2
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9))])
    near = np.concatenate([near, -near, np.array([0.0, -0.0, 1e-30, -1e-30, 7.0, -7.0, 1e30], np.float32)])
    return np.concatenate([all_bf16_as_f32(), grid, near]).astype(np.float32)


def test_e2m1_matches_oracle(sk):
    v = e2m1_probe_inputs()
    got = sk.convert_probe(0, torch.from_numpy(v).cuda()).cpu().numpy()
    want = np.array([oracle.e2m1_from_float(float(x)) for x in v], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), int(got[i]), int(want[i])) for i in bad[:8]]


def test_e4m3_matches_oracle(sk):
    lut = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    fin = np.unique(np.abs(lut[np.isfinite(lut)]))
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    extra = np.array([448, 464, 470, 480, 1e6, 2.0 ** -10, 2.0 ** -11, 0.0, -0.0], np.float32)
    v = np.concatenate([all_bf16_as_f32(), near, -near, extra, -extra]).astype(np.float32)
    got = sk.convert_probe(1, torch.from_numpy(v).cuda()).cpu().numpy()
    want = np.array([oracle.e4m3_from_float(float(x)) for x in v], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), int(got[i]), int(want[i])) for i in bad[:8]]


def test_e4m3_widening_is_exact(sk):
    b = np.array([i for i in range(256) if (i & 0x7F) != 0x7F], np.uint8)
    got = sk.convert_probe(3, torch.from_numpy(b).cuda()).cpu().numpy()
    want = np.array([oracle.e4m3_to_float(int(i)) for i in b], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_bf16_rounding_matches_oracle(sk):
    rng = np.random.default_rng(0)
    base = rng.integers(0, 0x7F7F, 200000).astype(np.uint32) << 16
    mids = base | 0x8000
    v = np.concatenate([base, mids, mids + 1, mids - 1,
                        rng.standard_normal(100000).astype(np.float32).view(np.uint32)]).view(np.float32)
    v = np.concatenate([v, -v])
    got = sk.convert_probe(2, torch.from_numpy(v).cuda()).cpu().numpy().view(np.uint16)
    sample = rng.choice(len(v), 40000, replace=False)
    want = np.array([oracle.bf16_from_double(float(v[i])) for i in sample], np.uint16)
    assert np.array_equal(got[sample], want)
    # and the full set against torch's own cast
    t = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, t)
