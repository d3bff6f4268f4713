"""Failure reporting without a GPU fault: a kernel whose bounded wait on an
mbarrier that nothing completes runs out sets its bit in the library's device
status word and returns; the host reads the bit, clears it, and the context
keeps computing correct results. (Every wait in the library's kernels is
bounded the same way.)"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_sm_skinny_gb300 import synth
from parity import check_gemm

pytestmark = pytest.mark.gpu


def test_wait_runs_out_sets_status_and_context_stays_usable():
    import nvfp4_sm_skinny_gb300 as sk

    assert sk.device_status(clear=True) == 0
    sk.wait_probe(2000)                        # 2 ms of waiting, then the kernel returns
    st = sk.device_status(clear=True)
    assert st & sk.SK_DEVICE_WAIT_PROBE
    assert sk.device_status(clear=True) == 0   # cleared
    x = synth.normal_bf16((4, 1024), 1.0, 5)
    w = synth.normal_bf16((256, 1024), 0.02, 6)
    y = sk.gemm_bf16(x.to("cuda"), w.to("cuda"))
    torch.cuda.synchronize()
    xb, wb = synth.bits(x), synth.bits(w)
    acc, absacc = oracle.gemm_f64(xb, wb)
    check_gemm(synth.bits(y), oracle.gemm_bf16(xb, wb), acc, absacc, 1024, sk.gemm_splits(4, 256, 1024))
    assert sk.device_status(clear=True) == 0


def test_wait_probe_rejects_bad_limits():
    import nvfp4_sm_skinny_gb300 as sk

    with pytest.raises(ValueError):
        sk.wait_probe(0)
    with pytest.raises(ValueError):
        sk.wait_probe(200000)
