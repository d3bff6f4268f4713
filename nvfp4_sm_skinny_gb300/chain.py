"""The per-layer decode chain of the hot path, wired from the public calls.

One layer, at M token rows (HIDDEN H = 8192, POOLED P = 4096):

    partial = h_l @ W_o^T                 o_proj      [8192, 8192]   (sk_gemm_dual_norm)
    s, u    = dual_norm(partial, s)       attention boundary, FP32 residual s in place
    a, a_sf, z = nvfp4(rmsnorm(u @ W_p^T)) pooler     [4096, 8192]   (sk_gemm_rmsnorm_nvfp4)
    h_{l+1} = z @ W_u^T                   unpooler    [8192, 4096]   (sk_gemm_bf16)

The routed experts between the pooler and the unpooler are outside this
path, so the unpooler reads the expert input z in their place (the order of
the pages: o_proj -> attention boundary -> pooler -> experts -> unpooler ->
next boundary). This module only allocates buffers and calls the binding;
every step runs in libsk's kernels. ``capture()`` records one pass into a
CUDA graph (the calls allocate nothing and are capturable).
"""
from __future__ import annotations

import copy

import torch

import nvfp4_sm_skinny_gb300 as sk
from nvfp4_sm_skinny_gb300 import synth

H = synth.HIDDEN
P = synth.POOLED


def layer_bytes(m: int) -> dict:
    """Algorithmic bytes of one layer (each input read once, each output
    written once; internal round trips such as the o_proj partial and the
    pooler's pre-norm y are not counted)."""
    oproj = 2 * H * H + 2 * m * H + 2 * m * H + 3 * 2 * H + 2 * 4 * m * H
    pooler = 2 * P * H + 2 * m * H + 2 * P + 4 + m * P // 2 + m * P // 16 + 2 * m * P
    unpooler = 2 * H * P + 2 * m * P + 2 * m * H
    return dict(oproj_dual=oproj, pooler_nvfp4=pooler, unpooler=unpooler,
                total=oproj + pooler + unpooler)


def gemm_bytes(m: int) -> int:
    """Algorithmic bytes of the three GEMMs of one layer taken alone."""
    return (2 * H * H + 2 * m * H + 2 * m * H) + (2 * P * H + 2 * m * H + 2 * m * P) + \
        (2 * H * P + 2 * m * P + 2 * m * H)


class DecodeChain:
    """Weights and buffers of an L-layer chain at M rows on one device."""

    def __init__(self, layers: int = 48, m: int = 16, device="cuda", eps: float = synth.EPS,
                 gain_center: float = synth.GAIN_CENTER, splits: int = 0,
                 prefetch_next: bool = True):
        self.L, self.m, self.device = layers, m, torch.device(device)
        # each GEMM starts the next GEMM's first weight stages towards L2
        self.prefetch_next = prefetch_next
        self.eps, self.gc, self.splits = eps, gain_center, splits
        dev = self.device
        self.w_o, self.w_p, self.w_u = [], [], []
        self.post_w, self.pre_w, self.beta, self.norm_w = [], [], [], []
        for l in range(layers):
            self.w_o.append(synth.chain_weight(l, 0, (H, H), device=dev))
            self.w_p.append(synth.chain_weight(l, 1, (P, H), device=dev))
            self.w_u.append(synth.chain_weight(l, 2, (H, P), device=dev))
            self.post_w.append(synth.chain_weight(l, 3, (H,), std=0.1, mean=1.0, device=dev))
            self.pre_w.append(synth.chain_weight(l, 4, (H,), std=0.1, mean=1.0, device=dev))
            self.beta.append(synth.chain_beta(l, device=dev))
            self.norm_w.append(synth.chain_weight(l, 6, (P,), std=0.1, device=dev))
        self.alpha = 1.0
        self.gs = torch.full((layers, 1), 448.0, dtype=torch.float32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.h = torch.zeros(layers + 1, m, H, **bf)           # h[0] is the input
        self.s = torch.zeros(m, H, dtype=torch.float32, device=dev)
        self.u = torch.zeros(layers, m, H, **bf)               # dual-norm outputs
        self.z = torch.zeros(layers, m, P, **bf)               # normalised pooler rows
        self.a = torch.zeros(layers, m, P // 2, dtype=torch.uint8, device=dev)
        self.a_sf = torch.zeros(layers, m, P // 16, dtype=torch.uint8, device=dev)
        self.ws_o = torch.zeros(layers, sk.gemm_dual_norm_workspace(m, H), dtype=torch.uint8, device=dev)
        self.ws_p = torch.zeros(layers, sk.gemm_rmsnorm_nvfp4_workspace(m, P), dtype=torch.uint8,
                                device=dev)

    def twin(self) -> "DecodeChain":
        """A chain on the same weights and global scales with its own
        activation buffers and workspaces, so that two steps can be in flight
        (one copying its inputs in or results out while the other runs)."""
        t = copy.copy(self)
        for name in ("h", "s", "u", "z", "a", "a_sf", "ws_o", "ws_p"):
            setattr(t, name, torch.zeros_like(getattr(self, name)))
        return t

    def set_input(self, h0: torch.Tensor, s0: torch.Tensor) -> None:
        self.h[0].copy_(h0)
        self.s.copy_(s0)

    def layer_op(self, l: int, op: int, stream=None) -> None:
        """One of the layer's three calls: 0 o_proj + dual norm, 1 pooler +
        RMSNorm + NVFP4, 2 unpooler."""
        if op == 0:
            sk.gemm_dual_norm(self.h[l], self.w_o[l], self.s, self.post_w[l], self.alpha,
                              self.beta[l], self.pre_w[l], out=self.u[l], eps_post=self.eps,
                              eps_pre=self.eps, workspace=self.ws_o[l], splits=self.splits,
                              stream=stream)
        elif op == 1:
            sk.gemm_rmsnorm_nvfp4(self.u[l], self.w_p[l], self.norm_w[l], self.eps, self.gc,
                                  self.gs[l], a=self.a[l], a_sf=self.a_sf[l], z_out=self.z[l],
                                  workspace=self.ws_p[l], splits=self.splits, stream=stream)
        else:
            sk.gemm_bf16(self.z[l], self.w_u[l], out=self.h[l + 1], splits=self.splits,
                         stream=stream)

    def next_weight(self, l: int, op: int):
        """The weight of the GEMM after layer l's call `op` (None after the last)."""
        if op == 0:
            return self.w_p[l]
        if op == 1:
            return self.w_u[l]
        return self.w_o[l + 1] if l + 1 < self.L else None

    def layer(self, l: int, stream=None) -> None:
        for op in range(3):
            if self.prefetch_next:
                sk.gemm_prefetch_next(self.next_weight(l, op))
            self.layer_op(l, op, stream)

    def forward(self, stream=None) -> None:
        for l in range(self.L):
            self.layer(l, stream)

    def gemms_only(self, stream=None) -> None:
        """The chain's three GEMMs per layer without their epilogues (same
        shapes, weights and launch configuration), for timing the GEMM kernel."""
        hint = sk.gemm_prefetch_next if self.prefetch_next else (lambda w: None)
        for l in range(self.L):
            hint(self.next_weight(l, 0))
            sk.gemm_bf16(self.h[l], self.w_o[l], out=self.ws_o[l][: self.m * H * 2].view(
                torch.bfloat16).view(self.m, H), splits=self.splits, stream=stream)
            hint(self.next_weight(l, 1))
            sk.gemm_bf16(self.u[l], self.w_p[l], out=self.ws_p[l][: self.m * P * 2].view(
                torch.bfloat16).view(self.m, P), splits=self.splits, stream=stream)
            hint(self.next_weight(l, 2))
            sk.gemm_bf16(self.z[l], self.w_u[l], out=self.h[l + 1], splits=self.splits,
                         stream=stream)

    def calibrate(self, x_cal: torch.Tensor, s_cal: torch.Tensor) -> None:
        """Sets each layer's NVFP4 global scale to 448 * 6 / amax(z) of one
        calibration pass (set-up, outside any timed region)."""
        self.set_input(x_cal, s_cal)
        self.gs.fill_(1.0)
        for l in range(self.L):
            self.layer(l)
            amax = self.z[l].float().abs().amax()
            self.gs[l].copy_(2688.0 / amax.clamp_min(1e-30))
        torch.cuda.synchronize(self.device)

    def capture(self, fn=None) -> torch.cuda.CUDAGraph:
        """One pass recorded as a CUDA graph (run once eagerly first)."""
        fn = fn or self.forward
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        torch.cuda.synchronize(self.device)
        return g

    launches_per_layer = 5
    gemm_launches_per_layer = 3
