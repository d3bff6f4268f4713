"""GPU parity of sk_gemm_nvfp4w_bf16, the weight-only NVFP4 GEMM, against the
CPU oracle (oracle_gemm_nvfp4w). Not on the pages: the weight is held in the
NVFP4 byte layout of the pooler page's module docstring (cutedsl/moe/
pooler_gather), applied to W [n, k] along K. Covers every (code, scale) pair
through one-hot activations (exact), several tiles with ragged tails and every
split count, a full-size weight quantized on the GPU with sampled outputs,
zero and negative w_scale, and bitwise run-to-run reproducibility."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_sm_skinny_gb300 import synth
from parity import check_gemm

pytestmark = pytest.mark.gpu
DEV = "cuda"
W_SCALE_GAMMA = 2.0 ** -24   # the FP32 multiply by w_scale after the sum


@pytest.fixture(scope="module")
def sk():
    import nvfp4_sm_skinny_gb300 as sk

    sk.lib()
    return sk


@pytest.fixture(autouse=True)
def _no_device_errors(sk):
    yield
    assert sk.device_status(clear=True) == 0


def scale_t(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def random_weight(n, k, seed, scale_lo=0x20, scale_hi=0x48):
    g = np.random.default_rng(seed)
    wq = g.integers(0, 256, (n, k // 2), dtype=np.uint8)
    wsf = g.integers(scale_lo, scale_hi, (n, k // 16), dtype=np.uint8)
    return wq, wsf


def run(sk, x, wq, wsf, w_scale, splits=0):
    y = sk.gemm_nvfp4w(x.to(DEV), torch.from_numpy(wq).to(DEV), torch.from_numpy(wsf).to(DEV),
                       scale_t(w_scale), splits=splits)
    torch.cuda.synchronize()
    return synth.bits(y)


def test_every_code_and_scale_exact(sk):
    # Row r holds one finite e4m3 scale (all 254 of them, both signs, plus two
    # zero-scale rows) and every code in every 16-column block; one-hot rows of
    # x read each weight alone, so y = bf16(W[r, j]) exactly.
    scales = [b for b in range(256) if b not in (0x7F, 0xFF)] + [0x00, 0x80]
    n, k = len(scales), 256
    assert n == 256
    codes = (np.arange(k)[None, :] * 7 + np.arange(n)[:, None]) % 16
    wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    wsf = np.repeat(np.array(scales, np.uint8)[:, None], k // 16, axis=1)
    wq_d, wsf_d = torch.from_numpy(wq).to(DEV), torch.from_numpy(wsf).to(DEV)
    ws = scale_t(1.0)
    got = np.zeros((n, k), np.uint16)
    for c0 in range(0, k, 16):
        x = torch.zeros(16, k, dtype=torch.bfloat16)
        x[torch.arange(16), c0 + torch.arange(16)] = 1.0
        y = sk.gemm_nvfp4w(x.to(DEV), wq_d, wsf_d, ws)
        torch.cuda.synchronize()
        got[:, c0:c0 + 16] = synth.bits(y).T
    want = oracle.gemm_nvfp4w(synth.bits(torch.eye(k, dtype=torch.bfloat16)), wq, wsf, 1.0).T
    assert np.array_equal(got, want)


@pytest.mark.parametrize("m", [1, 3, 16])
@pytest.mark.parametrize("n,k", [(16, 256), (400, 1024), (1024, 4096)])
def test_shapes_all_splits(sk, m, n, k):
    wq, wsf = random_weight(n, k, 10 * n + k)
    x = synth.normal_bf16((m, k), 1.0, 3 + m)
    xb = synth.bits(x)
    yref, acc, absacc = oracle.gemm_nvfp4w(xb, wq, wsf, 0.03125, return_acc=True)
    for splits in (0, 1, 2, 4, 8, 16):
        if sk.gemm_nvfp4w_supported(m, n, k, splits) is not None:
            continue
        s = splits or sk.gemm_nvfp4w_splits(m, n, k)
        y = run(sk, x, wq, wsf, 0.03125, splits)
        check_gemm(y, yref, acc, absacc, k, s, gamma_extra=W_SCALE_GAMMA,
                   label=f"nvfp4w M={m} [{n},{k}] S={splits or f'auto({s})'}")


def test_full_size_weight_quantized_on_gpu(sk):
    # A BF16 weight [8192, 8192] ~ N(0, 0.02) quantized by sk_nvfp4_quantize
    # with gs = 448 * 6 / amax, then the GEMM at M = 16 with w_scale = 1/gs;
    # the oracle checks one output feature in 61.
    n = k = 8192
    w = synth.normal_bf16((n, k), 0.02, 77, device=DEV)
    gs = float(np.float32(2688.0 / w.float().abs().max().item()))
    wq, wsf = sk.nvfp4_quantize(w, scale_t(gs))
    w_scale = float(np.float32(1.0 / gs))
    x = synth.normal_bf16((16, k), 1.0, 78)
    y = synth.bits(sk.gemm_nvfp4w(x.to(DEV), wq, wsf, scale_t(w_scale)))
    torch.cuda.synchronize()
    rows = np.arange(0, n, 61)
    wq_h, wsf_h = wq.cpu().numpy(), wsf.cpu().numpy()
    yref, acc, absacc = oracle.gemm_nvfp4w(synth.bits(x), wq_h[rows], wsf_h[rows], w_scale,
                                           return_acc=True)
    check_gemm(y[:, rows], yref, acc, absacc, k, sk.gemm_nvfp4w_splits(16, n, k),
               gamma_extra=W_SCALE_GAMMA, label="nvfp4w M=16 [8192,8192] quantized, sampled 1/61")
    # the quantized weight is the oracle's NVFP4 of the same BF16 weight
    a_ref, sf_ref = oracle.nvfp4_quantize(synth.bits(w[rows]), gs)
    assert np.array_equal(wq_h[rows], a_ref) and np.array_equal(wsf_h[rows], sf_ref)


def test_zero_and_negative_w_scale(sk):
    wq, wsf = random_weight(256, 512, 5)
    x = synth.normal_bf16((4, 512), 1.0, 6)
    assert np.all(run(sk, x, wq, wsf, 0.0) == 0)
    y_pos = run(sk, x, wq, wsf, 0.25)
    y_neg = run(sk, x, wq, wsf, -0.25)
    flip = np.where(y_pos == 0, 0, y_pos ^ 0x8000)
    assert np.array_equal(y_neg, flip)


def test_rows_beyond_m_are_not_written(sk):
    m, n, k = 5, 144, 512
    wq, wsf = random_weight(n, k, 8)
    x = synth.normal_bf16((m, k), 1.0, 9).to(DEV)
    buf = torch.full((m + 2, n), 7.0, dtype=torch.bfloat16, device=DEV)
    sk.gemm_nvfp4w(x, torch.from_numpy(wq).to(DEV), torch.from_numpy(wsf).to(DEV), scale_t(1.0),
                   out=buf[:m], splits=2)
    torch.cuda.synchronize()
    assert torch.all(buf[m:] == 7.0)


def test_bitwise_reproducible_100_runs(sk):
    n, k = 4096, 8192
    wq, wsf = random_weight(n, k, 11)
    wq_d, wsf_d = torch.from_numpy(wq).to(DEV), torch.from_numpy(wsf).to(DEV)
    x = synth.normal_bf16((16, k), 1.0, 12).to(DEV)
    ws = scale_t(0.01)
    first = sk.gemm_nvfp4w(x, wq_d, wsf_d, ws)
    out = torch.empty_like(first)
    for _ in range(100):
        sk.gemm_nvfp4w(x, wq_d, wsf_d, ws, out=out)
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
