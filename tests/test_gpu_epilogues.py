"""GPU parity of the epilogues against the CPU oracle: the pre-expert RMSNorm +
NVFP4 (standalone, fused behind the pooler GEMM, and the quantizer alone on
the oracle's own z), and the attention-boundary dual norm (standalone and
fused behind the o_proj GEMM). Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_sm_skinny_gb300 import synth
from parity import bf16_to_f64, check_gemm, check_nvfp4_end_to_end, ulp_distance

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sk():
    import nvfp4_sm_skinny_gb300 as sk

    sk.lib()
    return sk


@pytest.fixture(autouse=True)
def _no_device_errors(sk):
    yield
    assert sk.device_status(clear=True) == 0


def gs_tensor(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def calibrated_gs(w, norm_w):
    """Global scale from a seeded calibration batch through the oracle pipeline:
    gs = 448 * 6 / amax(z_cal)."""
    x_cal = synth.normal_bf16((16, w.shape[1]), 1.0, 1000)
    y = oracle.gemm_bf16(synth.bits(x_cal), synth.bits(w))
    z = oracle.rmsnorm_bf16(y, synth.bits(norm_w), synth.EPS, synth.GAIN_CENTER)
    amax = float(np.max(np.abs(bf16_to_f64(z))))
    return float(np.float32(2688.0 / amax))


# ----------------------------------------------------------- NVFP4 alone ----
@pytest.mark.parametrize("m,n,gs", [(1, 16, 1.0), (3, 4096, 500.0), (16, 4096, 2688.0 / 5),
                                    (7, 1024, 1e4), (2, 160, 1e-3)])
def test_quantize_bit_exact_on_oracle_z(sk, m, n, gs):
    g = torch.Generator().manual_seed(m * n)
    z = (torch.randn(m, n, generator=g) * torch.exp(torch.randn(m, 1, generator=g))).to(torch.bfloat16)
    z[0, :16] = 0.0                                     # an all-zero block
    if n >= 64:
        z[-1, 32:48] = -z[-1, 32:48].abs() * 1e-4        # tiny negatives
    zb = synth.bits(z)
    zb = np.where(zb == 0x8000, 0, zb)
    a_ref, sf_ref = oracle.nvfp4_quantize(zb, gs)
    a, a_sf = sk.nvfp4_quantize(synth.from_bits(zb, DEV), gs_tensor(gs))
    torch.cuda.synchronize()
    assert np.array_equal(a_sf.cpu().numpy(), sf_ref)
    assert np.array_equal(a.cpu().numpy(), a_ref)
    assert np.all(sf_ref[0, 0] == 0) and np.all(a_ref[0, :8] == 0)


# ---------------------------------------------------- RMSNorm + NVFP4 ----
@pytest.mark.parametrize("m,n", [(1, 4096), (8, 4096), (16, 4096), (4, 48), (16, 16384)])
def test_rmsnorm_nvfp4_standalone(sk, m, n):
    y = synth.normal_bf16((m, n), 1.8, 40 + m)
    w = synth.normal_bf16((n,), 0.1, 41)
    gs = 2688.0 / 7.0
    a, a_sf, z = sk.rmsnorm_nvfp4(y.to(DEV), w.to(DEV), synth.EPS, synth.GAIN_CENTER, gs_tensor(gs),
                                  z_out=True)
    torch.cuda.synchronize()
    z_ref = oracle.rmsnorm_bf16(synth.bits(y), synth.bits(w), synth.EPS, synth.GAIN_CENTER)
    d = ulp_distance(synth.bits(z), z_ref)
    assert d.max() <= 1 and (d != 0).mean() < 1e-3
    # NVFP4 decisions: bit-exact given the GPU's own z
    a_ref, sf_ref = oracle.nvfp4_quantize(synth.bits(z), gs)
    assert np.array_equal(a.cpu().numpy(), a_ref) and np.array_equal(a_sf.cpu().numpy(), sf_ref)
    # end to end against the oracle's own z
    a_ref2, sf_ref2 = oracle.nvfp4_quantize(z_ref, gs)
    check_nvfp4_end_to_end(a.cpu().numpy(), a_sf.cpu().numpy(), synth.bits(z), a_ref2, sf_ref2, z_ref)


def test_rmsnorm_zero_row_gives_zero_scale_and_codes(sk):
    y = torch.zeros(2, 4096, dtype=torch.bfloat16, device=DEV)
    w = synth.normal_bf16((4096,), 0.1, 41).to(DEV)
    a, a_sf, z = sk.rmsnorm_nvfp4(y, w, synth.EPS, 1.0, gs_tensor(300.0), z_out=True)
    torch.cuda.synchronize()
    assert torch.all(a == 0) and torch.all(a_sf == 0) and torch.all(z.view(torch.int16) == 0)


@pytest.mark.parametrize("b", [1, 8, 16])
def test_pooler_gemm_rmsnorm_nvfp4(sk, b):
    d = synth.pooler(b)
    gs = calibrated_gs(d["w"], d["norm_w"])
    a, a_sf, z, ws = sk.gemm_rmsnorm_nvfp4(d["x"].to(DEV), d["w"].to(DEV), d["norm_w"].to(DEV),
                                           d["eps"], d["gain_center"], gs_tensor(gs), z_out=True)
    torch.cuda.synchronize()
    y_gpu = ws[: b * 4096 * 2].view(torch.bfloat16).view(b, 4096)
    yb = synth.bits(y_gpu)
    # 1. the GEMM
    xb, wb = synth.bits(d["x"]), synth.bits(d["w"])
    acc, absacc = oracle.gemm_f64(xb, wb)
    y_ref = oracle.gemm_bf16(xb, wb)
    check_gemm(yb, y_ref, acc, absacc, 8192, sk.gemm_splits(b, 4096, 8192),
               label=f"pooler b={b} [4096,8192]")
    # 2. the norm of the GPU's own y
    z_tf = oracle.rmsnorm_bf16(yb, synth.bits(d["norm_w"]), d["eps"], d["gain_center"])
    zd = ulp_distance(synth.bits(z), z_tf)
    assert zd.max() <= 1
    # 3. NVFP4 of the GPU's own z: bit-exact
    a_tf, sf_tf = oracle.nvfp4_quantize(synth.bits(z), gs)
    assert np.array_equal(a.cpu().numpy(), a_tf) and np.array_equal(a_sf.cpu().numpy(), sf_tf)
    # 4. end to end from x
    a_ref, sf_ref, z_ref, _ = oracle.gemm_rmsnorm_nvfp4(xb, wb, synth.bits(d["norm_w"]), d["eps"],
                                                        d["gain_center"], gs)
    check_nvfp4_end_to_end(a.cpu().numpy(), a_sf.cpu().numpy(), synth.bits(z), a_ref, sf_ref, z_ref)


def test_pooler_saturates_beyond_calibration(sk):
    d = synth.pooler(4)
    gs = calibrated_gs(d["w"], d["norm_w"]) * 8      # scale too large: many blocks saturate
    a, a_sf, z, _ = sk.gemm_rmsnorm_nvfp4(d["x"].to(DEV), d["w"].to(DEV), d["norm_w"].to(DEV),
                                          d["eps"], d["gain_center"], gs_tensor(gs), z_out=True)
    torch.cuda.synchronize()
    a_tf, sf_tf = oracle.nvfp4_quantize(synth.bits(z), gs)
    assert np.array_equal(a.cpu().numpy(), a_tf) and np.array_equal(a_sf.cpu().numpy(), sf_tf)
    assert (sf_tf == 0x7E).any()


# ----------------------------------------------------- BF16 edge layers ----
@pytest.mark.parametrize("m,n", [(1, 4096), (5, 1024), (16, 4096), (3, 16), (2, 16384)])
def test_rmsnorm_bf16_standalone(sk, m, n):
    g = torch.Generator().manual_seed(31 * m + n)
    y = (torch.randn(m, n, generator=g) * 2.0).to(torch.bfloat16)
    y[0, :] = 0.0 if m > 1 else y[0, :]                 # an all-zero row gives zero rows out
    nw = (0.1 * torch.randn(n, generator=g)).to(torch.bfloat16)
    z = sk.rmsnorm_bf16(y.to(DEV), nw.to(DEV), synth.EPS, synth.GAIN_CENTER)
    torch.cuda.synchronize()
    z_ref = oracle.rmsnorm_bf16(synth.bits(y), synth.bits(nw), synth.EPS, synth.GAIN_CENTER)
    assert ulp_distance(synth.bits(z), z_ref).max() <= 1
    if m > 1:
        assert torch.all(z[0].view(torch.int16) == 0)


@pytest.mark.parametrize("b", [1, 16])
def test_pooler_edge_layer_bf16(sk, b):
    d = synth.pooler(b)
    x, w, nw = d["x"].to(DEV), d["w"].to(DEV), d["norm_w"].to(DEV)
    z, ws = sk.gemm_rmsnorm_bf16(x, w, nw, d["eps"], d["gain_center"])
    torch.cuda.synchronize()
    yb = synth.bits(ws[: b * 4096 * 2].view(torch.bfloat16).view(b, 4096))
    xb, wb = synth.bits(d["x"]), synth.bits(d["w"])
    acc, absacc = oracle.gemm_f64(xb, wb)
    check_gemm(yb, oracle.gemm_bf16(xb, wb), acc, absacc, 8192, sk.gemm_splits(b, 4096, 8192))
    z_tf = oracle.rmsnorm_bf16(yb, synth.bits(d["norm_w"]), d["eps"], d["gain_center"])
    assert ulp_distance(synth.bits(z), z_tf).max() <= 1
    # the same GEMM and norm as the NVFP4 layer's z
    _, _, z_nv, _ = sk.gemm_rmsnorm_nvfp4(x, w, nw, d["eps"], d["gain_center"], gs_tensor(300.0),
                                         z_out=True)
    torch.cuda.synchronize()
    assert torch.equal(z.view(torch.int16), z_nv.view(torch.int16))


# --------------------------------------------------------------- dual norm ----
def _check_dual(sk, d, p_bits, s0, s_gpu, out_gpu, post_w):
    s_ref, out_ref = oracle.dual_norm(p_bits, s0, None if post_w is None else synth.bits(post_w),
                                      d["alpha"], synth.bits(d["beta"]), synth.bits(d["pre_w"]),
                                      d["eps"], d["eps"])
    # FP32 residual: 1e-5 relative to the summands alpha*s and beta*q
    q_mag = np.abs(s_ref.astype(np.float64) - d["alpha"] * s0.astype(np.float64))
    tol = 1e-5 * (np.abs(d["alpha"] * s0.astype(np.float64)) + q_mag + 1e-30)
    err = np.abs(s_gpu.astype(np.float64) - s_ref.astype(np.float64))
    assert np.all(err <= tol), float(np.max(err / tol))
    # output: the pre-FFN norm of the GPU's own stream, within one BF16 ulp
    zero_beta = np.zeros(s0.shape[1], np.uint16)
    _, out_tf = oracle.dual_norm(np.zeros_like(p_bits), s_gpu, None, 1.0, zero_beta,
                                 synth.bits(d["pre_w"]), d["eps"], d["eps"])
    assert ulp_distance(synth.bits(out_gpu), out_tf).max() <= 1
    # and end to end against the oracle (cancellation in s makes a few
    # outputs differ by more than an ulp only where s ~ 0)
    dd = ulp_distance(synth.bits(out_gpu), out_ref)
    assert (dd > 1).mean() < 1e-3


@pytest.mark.parametrize("b", [1, 4, 16])
@pytest.mark.parametrize("with_post", [True, False])
def test_dual_norm_standalone(sk, b, with_post):
    d = synth.oproj_boundary(b)
    p = synth.normal_bf16((b, 8192), 1.5, 60 + b)
    post_w = d["post_w"] if with_post else None
    s_dev = d["stream"].to(DEV)
    out = sk.dual_norm_residual(p.to(DEV), s_dev, None if post_w is None else post_w.to(DEV),
                                d["alpha"], d["beta"].to(DEV), d["pre_w"].to(DEV),
                                eps_post=d["eps"], eps_pre=d["eps"])
    torch.cuda.synchronize()
    _check_dual(sk, d, synth.bits(p), d["stream"].numpy(), s_dev.cpu().numpy(), out, post_w)


def test_dual_norm_small_width_and_alpha(sk):
    g = torch.Generator().manual_seed(9)
    h = 72
    p = torch.randn(3, h, generator=g).to(torch.bfloat16)
    s = torch.randn(3, h, generator=g)
    beta = torch.rand(h, generator=g).to(torch.bfloat16)
    w1 = (1 + 0.1 * torch.randn(h, generator=g)).to(torch.bfloat16)
    w2 = (1 + 0.1 * torch.randn(h, generator=g)).to(torch.bfloat16)
    s_dev = s.to(DEV)
    out = sk.dual_norm_residual(p.to(DEV), s_dev, w1.to(DEV), 0.5, beta.to(DEV), w2.to(DEV),
                                eps_post=1e-5, eps_pre=1e-6, gc_post=0.25, gc_pre=0.5)
    torch.cuda.synchronize()
    s_ref, out_ref = oracle.dual_norm(synth.bits(p), s.numpy(), synth.bits(w1), 0.5, synth.bits(beta),
                                      synth.bits(w2), 1e-5, 1e-6, 0.25, 0.5)
    assert np.allclose(s_dev.cpu().numpy(), s_ref, rtol=1e-5, atol=1e-6)
    assert ulp_distance(synth.bits(out), out_ref).max() <= 1


@pytest.mark.parametrize("h", [8, 72, 1032, 4096, 8184])
def test_dual_norm_row_widths(sk, h):
    # widths that spread a row over 1, 2, 4 and 8 CTAs, with a partly idle last CTA
    g = torch.Generator().manual_seed(h)
    m = 5
    p = (torch.randn(m, h, generator=g) * 1.3).to(torch.bfloat16)
    s = torch.randn(m, h, generator=g)
    beta = (0.5 + torch.rand(h, generator=g)).to(torch.bfloat16)
    w1 = (1 + 0.1 * torch.randn(h, generator=g)).to(torch.bfloat16)
    w2 = (1 + 0.1 * torch.randn(h, generator=g)).to(torch.bfloat16)
    s_dev = s.to(DEV)
    out = sk.dual_norm_residual(p.to(DEV), s_dev, w1.to(DEV), 1.0, beta.to(DEV), w2.to(DEV))
    torch.cuda.synchronize()
    d = dict(alpha=1.0, beta=beta, pre_w=w2, eps=1e-6)
    _check_dual(sk, d, synth.bits(p), s.numpy(), s_dev.cpu().numpy(), out, w1)


@pytest.mark.parametrize("n", [16, 1040, 4112, 16368])
def test_rmsnorm_nvfp4_row_widths(sk, n):
    # widths that spread a row over 1, 3, 8 CTAs (ragged last CTA)
    m = 3
    y = synth.normal_bf16((m, n), 1.8, n)
    w = synth.normal_bf16((n,), 0.1, n + 1)
    gs = 2688.0 / 7.0
    a, a_sf, z = sk.rmsnorm_nvfp4(y.to(DEV), w.to(DEV), synth.EPS, synth.GAIN_CENTER, gs_tensor(gs),
                                  z_out=True)
    torch.cuda.synchronize()
    z_ref = oracle.rmsnorm_bf16(synth.bits(y), synth.bits(w), synth.EPS, synth.GAIN_CENTER)
    assert ulp_distance(synth.bits(z), z_ref).max() <= 1
    a_ref, sf_ref = oracle.nvfp4_quantize(synth.bits(z), gs)
    assert np.array_equal(a.cpu().numpy(), a_ref) and np.array_equal(a_sf.cpu().numpy(), sf_ref)


@pytest.mark.parametrize("b", [1, 4, 16])
def test_oproj_gemm_dual_norm(sk, b):
    d = synth.oproj_boundary(b)
    s_dev = d["stream"].to(DEV)
    out, ws = sk.gemm_dual_norm(d["x"].to(DEV), d["w"].to(DEV), s_dev, d["post_w"].to(DEV),
                                d["alpha"], d["beta"].to(DEV), d["pre_w"].to(DEV),
                                eps_post=d["eps"], eps_pre=d["eps"])
    torch.cuda.synchronize()
    p_gpu = synth.bits(ws[: b * 8192 * 2].view(torch.bfloat16).view(b, 8192))
    xb, wb = synth.bits(d["x"]), synth.bits(d["w"])
    acc, absacc = oracle.gemm_f64(xb, wb)
    check_gemm(p_gpu, oracle.gemm_bf16(xb, wb), acc, absacc, 1024, sk.gemm_splits(b, 8192, 1024),
               label=f"o_proj b={b} [8192,1024]")
    _check_dual(sk, d, p_gpu, d["stream"].numpy(), s_dev.cpu().numpy(), out, d["post_w"])


def test_epilogues_bitwise_reproducible(sk):
    # 100 repeated calls of each fused call give bitwise-identical outputs
    d = synth.pooler(16)
    x, w, nw = d["x"].to(DEV), d["w"].to(DEV), d["norm_w"].to(DEV)
    gs = gs_tensor(300.0)
    a0, s0, z0, ws0 = sk.gemm_rmsnorm_nvfp4(x, w, nw, d["eps"], 1.0, gs, z_out=True)
    a, s, z, ws = (torch.empty_like(a0), torch.empty_like(s0), torch.empty_like(z0),
                   torch.empty_like(ws0))
    for _ in range(100):
        sk.gemm_rmsnorm_nvfp4(x, w, nw, d["eps"], 1.0, gs, a=a, a_sf=s, z_out=z, workspace=ws)
        assert torch.equal(a, a0) and torch.equal(s, s0)
        assert torch.equal(z.view(torch.int16), z0.view(torch.int16))
    e = synth.oproj_boundary(16)
    xe, we = e["x"].to(DEV), e["w"].to(DEV)
    post_w, beta, pre_w = e["post_w"].to(DEV), e["beta"].to(DEV), e["pre_w"].to(DEV)
    base = e["stream"].to(DEV)
    s_dev = base.clone()
    out0, _ = sk.gemm_dual_norm(xe, we, s_dev, post_w, 1.0, beta, pre_w)
    s_ref = s_dev.clone()
    out = torch.empty_like(out0)
    for _ in range(100):
        s_dev.copy_(base)
        sk.gemm_dual_norm(xe, we, s_dev, post_w, 1.0, beta, pre_w, out=out)
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(s_dev, s_ref)
