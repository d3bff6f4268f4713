"""GPU parity of sk_gemm_bf16 against the CPU oracle (all calls go through the
C ABI via the binding). Covers exact special cases (identity and one-hot
weights, zeros), several tiles with a ragged tail, every split count, the
unpooler shard and the M x (N, K) sweep, the largest shapes (sampled), padding
rows, and bitwise run-to-run reproducibility."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_sm_skinny_gb300 import synth
from parity import check_gemm, ulp_distance

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


def run(sk, x, w, splits=0):
    y = sk.gemm_bf16(x.to(DEV), w.to(DEV), splits=splits)
    torch.cuda.synchronize()
    return synth.bits(y)


def ref(x, w):
    xb, wb = synth.bits(x), synth.bits(w)
    acc, absacc = oracle.gemm_f64(xb, wb)
    return oracle.gemm_bf16(xb, wb), acc, absacc


@pytest.mark.parametrize("k", [64, 128, 1024])
@pytest.mark.parametrize("splits", [1, 2])
def test_identity_weight_is_exact(sk, k, splits):
    if k % (64 * splits):
        pytest.skip("no such split")
    x = synth.normal_bf16((16, k), 1.0, 1)
    w = torch.eye(k, dtype=torch.bfloat16)
    y = run(sk, x, w, splits)
    xb = synth.bits(x)
    assert np.array_equal(y, np.where(xb == 0x8000, 0, xb))


def test_one_hot_power_of_two_weight_is_exact(sk):
    g = torch.Generator().manual_seed(3)
    n, k = 384, 512
    perm = torch.randint(0, k, (n,), generator=g)
    scale = 2.0 ** torch.randint(-3, 4, (n,), generator=g).float()
    w = torch.zeros(n, k)
    w[torch.arange(n), perm] = scale
    x = synth.normal_bf16((7, k), 1.0, 4)
    for splits in (1, 2, 4, 8):
        y = run(sk, x, w.to(torch.bfloat16), splits)
        want = (x.float()[:, perm] * scale[None]).to(torch.bfloat16)
        assert np.array_equal(y, synth.bits(want)), splits


@pytest.mark.parametrize("n,k", [(1024, 4096), (8192, 1024), (4096, 8192)])
def test_one_hot_weight_exact_on_auto_plans(sk, n, k):
    # The automatic plans of these shapes use 64-row tiles with split 4, 56-row
    # tiles (both with the 64-row MMA, whose accumulator rows sit in lanes
    # 32 * (r / 16) + r % 16) and 128-row tiles with split 4: with one
    # power-of-two weight per row every output is a single exact product, so
    # a row read from the wrong TMEM lane or stored to the wrong feature shows.
    g = torch.Generator().manual_seed(n + k)
    perm = torch.randint(0, k, (n,), generator=g)
    scale = 2.0 ** torch.randint(-3, 4, (n,), generator=g).float()
    w = torch.zeros(n, k, dtype=torch.bfloat16)
    w[torch.arange(n), perm] = scale.to(torch.bfloat16)
    x = synth.normal_bf16((16, k), 1.0, 9)
    y = run(sk, x, w, 0)
    want = (x.float()[:, perm] * scale[None]).to(torch.bfloat16)
    assert np.array_equal(y, synth.bits(want))


def test_zero_activations_give_positive_zero(sk):
    w = synth.normal_bf16((256, 512), 0.02, 5)
    for xval in (0.0, -0.0):
        x = torch.full((3, 512), xval, dtype=torch.bfloat16)
        assert np.all(run(sk, x, w, 2) == 0)


@pytest.mark.parametrize("m", [1, 3, 8, 16])
@pytest.mark.parametrize("n,k", [(16, 64), (144, 256), (400, 1024), (1024, 512)])
def test_small_shapes_all_splits(sk, m, n, k):
    x = synth.normal_bf16((m, k), 1.0, 10 + m)
    w = synth.normal_bf16((n, k), 0.02, 20 + n)
    yref, acc, absacc = ref(x, w)
    for splits in (1, 2, 4, 8, 16):
        if k % (64 * splits):
            continue
        y = run(sk, x, w, splits)
        check_gemm(y, yref, acc, absacc, k, splits, label=f"small M={m} [{n},{k}] S={splits}")


def test_unpooler_shard_m1(sk):
    # x [1, 4096] ~ N(0,1), W [1024, 4096] ~ N(0, 0.02), auto split count
    x, w = synth.unpooler_shard()
    yref, acc, absacc = ref(x, w)
    s = sk.gemm_splits(1, 1024, 4096)
    y = run(sk, x, w)
    check_gemm(y, yref, acc, absacc, 4096, s, label=f"unpooler shard M=1 [1024,4096] S={s}")
    assert ulp_distance(y, yref).max() <= 1


@pytest.mark.parametrize("n,k", [(1024, 4096), (8192, 4096)])
def test_sweep_m_and_splits(sk, n, k):
    w = synth.gemm_weight(n, k, copy=0)
    wd = w.to(DEV)
    for m in (1, 2, 4, 8, 16):
        x = synth.gemm_x(m, k)
        yref, acc, absacc = ref(x, w)
        for splits in (0, 1, 2, 4, 8):
            y = sk.gemm_bf16(x.to(DEV), wd, splits=splits)
            torch.cuda.synchronize()
            s = splits or sk.gemm_splits(m, n, k)
            check_gemm(synth.bits(y), yref, acc, absacc, k, s,
                       label=f"sweep M={m} [{n},{k}] S={splits or f'auto({s})'}")


@pytest.mark.parametrize("m,n,k", [(16, 24576, 2048), (4, 1024, 32768), (16, 8192, 16384)])
def test_large_shapes_sampled(sk, m, n, k):
    # more row tiles than SMs (a second wave), or a long K (many stages, up to
    # 16 slices); the oracle checks a sample of output features, one in 61
    x = synth.normal_bf16((m, k), 1.0, 40 + m)
    w = synth.normal_bf16((n, k), 0.02, 41 + n % 97)
    y = run(sk, x, w)
    cols = np.arange(0, n, 61)
    yref, acc, absacc = ref(x, w[torch.as_tensor(cols)])
    check_gemm(y[:, cols], yref, acc, absacc, k, sk.gemm_splits(m, n, k),
               label=f"large M={m} [{n},{k}] sampled 1/61")


@pytest.mark.parametrize("n2,k2", [(4096, 8192), (1024, 512)])
def test_prefetch_hint_leaves_results_unchanged(sk, n2, k2):
    # A GEMM told which weight comes next starts that weight's first stages
    # towards L2 after its own last copy; the next GEMM then skips its own
    # look-ahead. Neither result may change, including when the hinted shape
    # is not the one that follows.
    x = synth.gemm_x(16, 4096).to(DEV)
    w = synth.gemm_weight(8192, 4096).to(DEV)
    w2 = synth.gemm_weight(n2, k2, 1).to(DEV)
    x2 = synth.gemm_x(16, k2).to(DEV)
    y_ref = sk.gemm_bf16(x, w)
    y2_ref = sk.gemm_bf16(x2, w2)
    for _ in range(3):
        sk.gemm_prefetch_next(w2)
        y = sk.gemm_bf16(x, w)
        y2 = sk.gemm_bf16(x2, w2)            # its first stages were warmed
        sk.gemm_prefetch_next(w)             # a hint that does not match what follows
        y3 = sk.gemm_bf16(x2, w2)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        assert torch.equal(y2.view(torch.int16), y2_ref.view(torch.int16))
        assert torch.equal(y3.view(torch.int16), y2_ref.view(torch.int16))
    sk.gemm_prefetch_next(None)


@pytest.mark.parametrize("m,n,k", [(1, 1024, 4096), (16, 8192, 4096), (5, 400, 1024)])
def test_x_ready_run_matches_plain_calls(sk, m, n, k):
    # A run of GEMMs on one input that no kernel writes: with x_ready each call
    # reads x at once and only its stores wait, so calls overlap. Each result
    # must equal the plain call's, bit for bit, and a shared output must end
    # holding the last call's result (stores stay in stream order).
    x = synth.gemm_x(m, k).to(DEV)
    ws = [synth.gemm_weight(n, k, 20 + i).to(DEV) for i in range(6)]
    torch.cuda.synchronize()
    ref = [sk.gemm_bf16(x, w) for w in ws]
    outs = [torch.empty(m, n, dtype=torch.bfloat16, device=DEV) for _ in ws]
    shared = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    for _ in range(3):
        for w, o in zip(ws, outs):
            sk.gemm_bf16(x, w, out=o, x_ready=True)
        for w in ws:
            sk.gemm_bf16(x, w, out=shared, x_ready=True)
        torch.cuda.synchronize()
        for r, o in zip(ref, outs):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
        assert torch.equal(shared.view(torch.int16), ref[-1].view(torch.int16))
    assert sk.device_status() == 0


def test_rows_beyond_m_are_not_written(sk):
    m, n, k = 5, 256, 256
    x = synth.normal_bf16((m, k), 1.0, 30)
    w = synth.normal_bf16((n, k), 0.02, 31)
    buf = torch.full((m + 2, n), 7.0, dtype=torch.bfloat16, device=DEV)
    sk.gemm_bf16(x.to(DEV), w.to(DEV), out=buf[:m], splits=2)
    torch.cuda.synchronize()
    assert torch.all(buf[m:] == 7.0)


def test_bitwise_reproducible_100_runs(sk):
    m, n, k = 16, 8192, 4096
    x = synth.gemm_x(m, k).to(DEV)
    w = synth.gemm_weight(n, k).to(DEV)
    for splits in (0, 4):
        first = sk.gemm_bf16(x, w, splits=splits)
        out = torch.empty_like(first)
        for _ in range(100):
            sk.gemm_bf16(x, w, out=out, splits=splits)
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    # the small single-tile shape at the largest split count
    x1, w1 = synth.unpooler_shard()
    x1, w1 = x1.to(DEV), w1.to(DEV)
    first = sk.gemm_bf16(x1, w1, splits=16)
    for _ in range(100):
        assert torch.equal(sk.gemm_bf16(x1, w1, splits=16).view(torch.int16), first.view(torch.int16))


def test_invalid_arguments_raise(sk):
    x = torch.zeros(17, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        sk.gemm_bf16(x, w)
    with pytest.raises(ValueError):
        sk.gemm_bf16(x[:4], w, splits=3)
