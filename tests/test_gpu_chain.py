"""The decode chain at full size in the launch configuration bench.py times
(M = 16, automatic split counts, CUDA-graph replay): each sampled layer is
checked against the oracle fed that layer's GPU inputs (teacher forcing), and
the graph replay must equal the eager calls bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_sm_skinny_gb300 import synth
from parity import check_gemm, check_nvfp4_end_to_end, ulp_distance

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def chain():
    import nvfp4_sm_skinny_gb300 as sk
    from nvfp4_sm_skinny_gb300.chain import DecodeChain

    c = DecodeChain(layers=48, m=16, device=DEV)
    h0 = synth.normal_bf16((16, synth.HIDDEN), 1.0, 0).to(DEV)
    s0 = synth.normal_f32((16, synth.HIDDEN), 503).to(DEV)
    c.calibrate(synth.normal_bf16((16, synth.HIDDEN), 1.0, 1000).to(DEV), s0)
    c.set_input(h0, s0)
    c.h0, c.s0 = h0, s0
    yield c
    assert sk.device_status() == 0


def check_layer(c, l, s_before):
    H, P = synth.HIDDEN, synth.POOLED
    b = synth.bits
    m = c.m
    xb, wo = b(c.h[l]), b(c.w_o[l])
    # o_proj partial
    part = b(c.ws_o[l][: m * H * 2].view(torch.bfloat16).view(m, H))
    acc, absacc = oracle.gemm_f64(xb, wo)
    check_gemm(part, oracle.gemm_bf16(xb, wo), acc, absacc, H, _splits(m, H, H),
               label=f"chain M={m} layer {l} o_proj [8192,8192]")
    # dual norm on the GPU's partial and the stream before this layer
    s_ref, u_ref = oracle.dual_norm(part, s_before, b(c.post_w[l]), c.alpha, b(c.beta[l]),
                                    b(c.pre_w[l]), c.eps, c.eps)
    s_gpu = c.s_after[l]
    q_mag = np.abs(s_ref.astype(np.float64) - s_before.astype(np.float64))
    tol = 1e-5 * (np.abs(s_before.astype(np.float64)) + q_mag + 1e-30)
    assert np.all(np.abs(s_gpu.astype(np.float64) - s_ref) <= tol)
    assert (ulp_distance(b(c.u[l]), u_ref) > 1).mean() < 1e-3
    # pooler + RMSNorm + NVFP4 on the GPU's u
    ub, wp = b(c.u[l]), b(c.w_p[l])
    y = b(c.ws_p[l][: m * P * 2].view(torch.bfloat16).view(m, P))
    acc, absacc = oracle.gemm_f64(ub, wp)
    check_gemm(y, oracle.gemm_bf16(ub, wp), acc, absacc, H, _splits(m, P, H),
               label=f"chain M={m} layer {l} pooler [4096,8192]")
    gs = float(c.gs[l].item())
    z_tf = oracle.rmsnorm_bf16(y, b(c.norm_w[l]), c.eps, c.gc)
    assert ulp_distance(b(c.z[l]), z_tf).max() <= 1
    a_tf, sf_tf = oracle.nvfp4_quantize(b(c.z[l]), gs)
    assert np.array_equal(c.a[l].cpu().numpy(), a_tf) and np.array_equal(c.a_sf[l].cpu().numpy(), sf_tf)
    a_ref, sf_ref, z_ref, _ = oracle.gemm_rmsnorm_nvfp4(ub, wp, b(c.norm_w[l]), c.eps, c.gc, gs)
    check_nvfp4_end_to_end(c.a[l].cpu().numpy(), c.a_sf[l].cpu().numpy(), b(c.z[l]), a_ref, sf_ref,
                           z_ref)
    # unpooler on the GPU's z
    zb, wu = b(c.z[l]), b(c.w_u[l])
    acc, absacc = oracle.gemm_f64(zb, wu)
    check_gemm(b(c.h[l + 1]), oracle.gemm_bf16(zb, wu), acc, absacc, P, _splits(m, H, P),
               label=f"chain M={m} layer {l} unpooler [8192,4096]")


def _splits(m, n, k):
    import nvfp4_sm_skinny_gb300 as sk

    return sk.gemm_splits(m, n, k)


def test_chain_sampled_layers_match_oracle(chain):
    c = chain
    sampled = (0, 1, 24, 47)
    c.s_after = {}
    s_before = {}
    for l in range(c.L):
        if l in sampled:
            s_before[l] = c.s.cpu().numpy().copy()
        c.layer(l)
        if l in sampled:
            torch.cuda.synchronize()
            c.s_after[l] = c.s.cpu().numpy().copy()
    torch.cuda.synchronize()
    for l in sampled:
        check_layer(c, l, s_before[l])


def test_graph_replay_equals_eager(chain):
    c = chain
    c.set_input(c.h0, c.s0)
    c.forward()
    torch.cuda.synchronize()
    eager = (c.h[c.L].clone(), c.a.clone(), c.a_sf.clone(), c.s.clone())
    g = c.capture(c.forward)          # runs once eagerly, then captures
    for _ in range(100):
        c.set_input(c.h0, c.s0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(c.h[c.L].view(torch.int16), eager[0].view(torch.int16))
        assert torch.equal(c.a, eager[1]) and torch.equal(c.a_sf, eager[2])
        assert torch.equal(c.s, eager[3])


def test_prefetch_hints_leave_the_chain_unchanged(chain):
    # forward() hints each GEMM with the next GEMM's weight; without the hints
    # every result is the same, bit for bit
    c = chain
    assert c.prefetch_next
    c.set_input(c.h0, c.s0)
    c.forward()
    torch.cuda.synchronize()
    hinted = (c.h[c.L].clone(), c.a.clone(), c.a_sf.clone(), c.s.clone(), c.u.clone())
    c.prefetch_next = False
    try:
        c.set_input(c.h0, c.s0)
        c.forward()
        torch.cuda.synchronize()
    finally:
        c.prefetch_next = True
    assert torch.equal(c.h[c.L].view(torch.int16), hinted[0].view(torch.int16))
    assert torch.equal(c.a, hinted[1]) and torch.equal(c.a_sf, hinted[2])
    assert torch.equal(c.s, hinted[3])
    assert torch.equal(c.u.view(torch.int16), hinted[4].view(torch.int16))


@pytest.mark.parametrize("m", [1, 3])
def test_small_m_chain_matches_oracle(m):
    # the same chain at a ragged token count (rows past m are zero-filled by the
    # copy engine and never stored), every layer checked against the oracle on
    # its GPU inputs, with the next-weight hints on
    import nvfp4_sm_skinny_gb300 as sk
    from nvfp4_sm_skinny_gb300.chain import DecodeChain

    c = DecodeChain(layers=3, m=m, device=DEV)
    assert c.prefetch_next
    h0 = synth.normal_bf16((m, synth.HIDDEN), 1.0, 7).to(DEV)
    s0 = synth.normal_f32((m, synth.HIDDEN), 8).to(DEV)
    c.calibrate(synth.normal_bf16((m, synth.HIDDEN), 1.0, 9).to(DEV), s0)
    c.set_input(h0, s0)
    c.s_after = {}
    for l in range(c.L):
        s_before = c.s.cpu().numpy().copy()
        c.layer(l)
        torch.cuda.synchronize()
        c.s_after[l] = c.s.cpu().numpy().copy()
        check_layer(c, l, s_before)
    assert sk.device_status() == 0
