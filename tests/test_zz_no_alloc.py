"""sk_gemm_rmsnorm_nvfp4_static: the pooler call for callers that cannot
allocate device memory (a plugin enqueue handed no workspace, a serving loop
with a fixed memory budget). Its GEMM output
lives in the library's static device scratch instead of a workspace.

Called here through the C ABI (ctypes) on two calls in a row with different
inputs and compared with the workspace entry point sk_gemm_rmsnorm_nvfp4: the
same kernels in the same launch configuration, so the NVFP4 codes, scales and
the normalised rows must agree bit for bit -- the tolerance the parity tests
use for NVFP4 decisions on identical inputs. This file is collected last so a
run that stops at the first failure has run every other test first; it also
passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from nvfp4_sm_skinny_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_scratch_entry_matches_workspace_entry():
    import nvfp4_sm_skinny_gb300 as sk

    lib = sk.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (b, n, k) in enumerate([(16, 4096, 8192), (5, 1024, 4096)]):
        x = synth.normal_bf16((b, k), 1.0, 700 + call).to(DEV)
        w = synth.normal_bf16((n, k), 0.02, 710 + call).to(DEV)
        norm_w = synth.normal_bf16((n,), 0.1, 720 + call).to(DEV)
        gs = torch.tensor([300.0 + call], dtype=torch.float32, device=DEV)

        a_ref, sf_ref, z_ref, _ = sk.gemm_rmsnorm_nvfp4(x, w, norm_w, synth.EPS, synth.GAIN_CENTER, gs,
                                                        z_out=True)
        a = torch.full((b, n // 2), 0xAB, dtype=torch.uint8, device=DEV)
        a_sf = torch.full((b, n // 16), 0xAB, dtype=torch.uint8, device=DEV)
        z = torch.zeros(b, n, dtype=torch.bfloat16, device=DEV)
        st = lib.sk_gemm_rmsnorm_nvfp4_static(_ptr(x), _ptr(w), _ptr(norm_w), synth.EPS,
                                               synth.GAIN_CENTER, _ptr(gs), _ptr(a), _ptr(a_sf),
                                               _ptr(z), b, n, k, 0, stream)
        assert st == 0, sk.last_error()
        torch.cuda.synchronize()
        assert torch.equal(a, a_ref), f"call {call}: codes differ"
        assert torch.equal(a_sf, sf_ref), f"call {call}: scales differ"
        assert torch.equal(z.view(torch.int16), z_ref.view(torch.int16)), f"call {call}: z differs"
    assert sk.device_status() == 0


def test_static_scratch_rejects_shapes_beyond_its_size():
    import nvfp4_sm_skinny_gb300 as sk

    lib = sk.lib()
    fake = ctypes.c_void_p(1 << 20)
    # 16 x 16384 BF16 needs 512 KiB > 256 KiB of static scratch
    st = lib.sk_gemm_rmsnorm_nvfp4_static(fake, fake, fake, 1e-6, 1.0, fake, fake, fake, None,
                                           16, 16384, 4096, 0, None)
    assert st == sk.SK_ERR_INVALID_ARG
    assert "static scratch" in sk.last_error()
