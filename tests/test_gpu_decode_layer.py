"""GPU parity of sk_decode_layer, the whole decode layer in one persistent
kernel: every stage is checked against the oracle fed the kernel's own inputs
to that stage (teacher forcing, through the optional partial / pooler-row
outputs), at full size (M = 16, HIDDEN 8192, POOLED 4096) and on small ragged
shapes; results are bitwise reproducible and agree with the separate calls."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_sm_skinny_gb300 import synth
from parity import check_gemm, check_nvfp4_end_to_end, ulp_distance

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


def check_stages(m, h_in, w_o, w_p, w_u, s0, post_w, alpha, beta, pre_w, norm_w, gs, eps, gc,
                 p_gpu, s_gpu, u_gpu, y_gpu, z_gpu, a_gpu, sf_gpu, h_gpu):
    b = synth.bits
    H, Ko = w_o.shape
    P = w_p.shape[0]
    # o_proj partial
    xb, wb = b(h_in), b(w_o)
    acc, absacc = oracle.gemm_f64(xb, wb)
    check_gemm(p_gpu, oracle.gemm_bf16(xb, wb), acc, absacc, Ko, 1)
    # dual norm on the GPU's partial
    s_ref, u_ref = oracle.dual_norm(p_gpu, s0, None if post_w is None else b(post_w), alpha, b(beta),
                                    b(pre_w), eps, eps)
    q_mag = np.abs(s_ref.astype(np.float64) - alpha * s0.astype(np.float64))
    tol = 1e-5 * (np.abs(alpha * s0.astype(np.float64)) + q_mag + 1e-30)
    assert np.all(np.abs(s_gpu.astype(np.float64) - s_ref) <= tol)
    _, u_tf = oracle.dual_norm(np.zeros_like(p_gpu), s_gpu, None, 1.0, np.zeros(H, np.uint16),
                               b(pre_w), eps, eps)
    assert ulp_distance(u_gpu, u_tf).max() <= 1
    # pooler GEMM on the GPU's u
    acc, absacc = oracle.gemm_f64(u_gpu, b(w_p))
    check_gemm(y_gpu, oracle.gemm_bf16(u_gpu, b(w_p)), acc, absacc, H, 1)
    z_tf = oracle.rmsnorm_bf16(y_gpu, b(norm_w), eps, gc)
    assert ulp_distance(z_gpu, z_tf).max() <= 1
    a_tf, sf_tf = oracle.nvfp4_quantize(z_gpu, gs)
    assert np.array_equal(a_gpu, a_tf) and np.array_equal(sf_gpu, sf_tf)
    a_ref, sf_ref = oracle.nvfp4_quantize(z_tf, gs)
    check_nvfp4_end_to_end(a_gpu, sf_gpu, z_gpu, a_ref, sf_ref, z_tf)
    # unpooler on the GPU's z
    acc, absacc = oracle.gemm_f64(z_gpu, b(w_u))
    check_gemm(h_gpu, oracle.gemm_bf16(z_gpu, b(w_u)), acc, absacc, P, 1)


def run_layer(sk, m, H, P, Ko, seed, with_post=True, gs_val=300.0):
    g = lambda shape, std, sd, mean=0.0: synth.normal_bf16(shape, std, seed + sd, mean=mean).to(DEV)
    h_in = g((m, Ko), 1.0, 0)
    w_o, w_p, w_u = g((H, Ko), 0.02, 1), g((P, H), 0.02, 2), g((H, P), 0.02, 3)
    post_w = g((H,), 0.1, 4, 1.0) if with_post else None
    pre_w, norm_w = g((H,), 0.1, 5, 1.0), g((P,), 0.1, 6)
    beta = synth.uniform_bf16((H,), 0.5, 1.5, seed + 7).to(DEV)
    s = synth.normal_f32((m, H), seed + 8).to(DEV)
    s0 = s.cpu().numpy().copy()
    gs = torch.tensor([gs_val], dtype=torch.float32, device=DEV)
    bf = dict(dtype=torch.bfloat16, device=DEV)
    u, z, hout = torch.empty(m, H, **bf), torch.empty(m, P, **bf), torch.empty(m, H, **bf)
    p_dbg, y_dbg = torch.empty(m, H, **bf), torch.empty(m, P, **bf)
    a = torch.empty(m, P // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(m, P // 16, dtype=torch.uint8, device=DEV)
    ws = torch.empty(sk.decode_layer_workspace(), dtype=torch.uint8, device=DEV)
    sk.decode_layer(h_in, w_o, w_p, w_u, s, post_w, 1.0, beta, pre_w, norm_w, gs, u, z, a, sf, hout,
                    ws, partial_out=p_dbg, y_out=y_dbg, eps_pool=1e-6, gc_pool=1.0)
    torch.cuda.synchronize()
    b = synth.bits
    check_stages(m, h_in, w_o, w_p, w_u, s0, post_w, 1.0, beta, pre_w, norm_w, gs_val, 1e-6, 1.0,
                 b(p_dbg), s.cpu().numpy(), b(u), b(y_dbg), b(z), a.cpu().numpy(), sf.cpu().numpy(),
                 b(hout))
    return dict(h_in=h_in, w_o=w_o, w_p=w_p, w_u=w_u, post_w=post_w, pre_w=pre_w, norm_w=norm_w,
                beta=beta, s0=s0, gs=gs, out=(b(hout), a.cpu().numpy(), sf.cpu().numpy(),
                                               s.cpu().numpy(), b(u), b(z)))


@pytest.mark.parametrize("m,H,P,Ko", [(3, 1024, 512, 1024), (16, 2048, 1024, 512), (1, 512, 256, 256),
                                      (5, 8192, 4096, 1024)])
def test_decode_layer_small_and_ragged(sk, m, H, P, Ko):
    run_layer(sk, m, H, P, Ko, seed=100 * m + H % 97)


def test_decode_layer_full_size_no_post_weight(sk):
    run_layer(sk, 16, 8192, 4096, 8192, seed=7, with_post=False)


def test_decode_layer_bitwise_reproducible(sk):
    r1 = run_layer(sk, 16, 8192, 4096, 8192, seed=11)
    r2 = run_layer(sk, 16, 8192, 4096, 8192, seed=11)
    for x, y in zip(r1["out"], r2["out"]):
        assert np.array_equal(x, y)


def test_decode_chain_fused_matches_oracle_and_separate_calls(sk):
    from nvfp4_sm_skinny_gb300.chain import DecodeChain

    c = DecodeChain(layers=3, m=16, device=DEV)
    h0 = synth.normal_bf16((16, synth.HIDDEN), 1.0, 0).to(DEV)
    s0 = synth.normal_f32((16, synth.HIDDEN), 503).to(DEV)
    c.calibrate(synth.normal_bf16((16, synth.HIDDEN), 1.0, 1000).to(DEV), s0)
    # separate calls
    c.set_input(h0, s0)
    c.forward()
    torch.cuda.synchronize()
    sep_h, sep_s = c.h[c.L].clone(), c.s.clone()
    # fused, with every stage teacher-forced
    c.keep_intermediates()
    c.set_input(h0, s0)
    b = synth.bits
    for l in range(c.L):
        s_before = c.s.cpu().numpy().copy()
        c.layer_fused(l)
        torch.cuda.synchronize()
        check_stages(16, c.h[l], c.w_o[l], c.w_p[l], c.w_u[l], s_before, c.post_w[l], c.alpha,
                     c.beta[l], c.pre_w[l], c.norm_w[l], float(c.gs[l].item()), c.eps, c.gc,
                     b(c.p_dbg[l]), c.s.cpu().numpy(), b(c.u[l]), b(c.y_dbg[l]), b(c.z[l]),
                     c.a[l].cpu().numpy(), c.a_sf[l].cpu().numpy(), b(c.h[l + 1]))
    # the fused and the separate paths agree closely after three layers
    fh, sh = c.h[c.L].float(), sep_h.float()
    rel = (fh - sh).norm() / sh.norm()
    assert rel < 2e-2, float(rel)
    g = c.capture(c.forward_fused)
    c.set_input(h0, s0)
    g.replay()
    torch.cuda.synchronize()
    first = c.h[c.L].clone()
    c.set_input(h0, s0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), c.h[c.L].view(torch.int16))


def test_decode_layer_rejects_bad_arguments(sk):
    t = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        sk.decode_layer(torch.zeros(17, 64, dtype=torch.bfloat16, device=DEV), t, t, t,
                        torch.zeros(17, 4, device=DEV), None, 1.0, t[0], t[0], t[0],
                        torch.ones(1, device=DEV), t, t, t, t, t,
                        torch.zeros(16, dtype=torch.uint8, device=DEV))
