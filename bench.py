"""Benchmark of the skinny-GEMM hot path on GB300.

One step = one pass of the 48-layer decode chain at M = 16 token rows, every
row of the hot path in each layer:

    o_proj GEMM [8192, 8192] + dual norm (post_attn_norm, gated FP32 residual,
    pre_ffn_norm) -> pooler GEMM [4096, 8192] + pre-expert RMSNorm + NVFP4 ->
    unpooler GEMM [8192, 4096]

with distinct seeded weights per layer (12 GiB, far larger than the 129 MB
L2, so no flush is needed between steps). The pass is captured once as a CUDA
graph of the C-ABI calls and replayed; kernels are chained with programmatic
dependent launch.

Reported: whole-job achieved HBM GB/s (algorithmic bytes / time) with the
spread of the step time, the dominant kernel's roofline (the skinny GEMM timed
alone over the same launches), the end-to-end rate with host buffers, the
single-call workloads (`per_config`: the M=1 unpooler shard, the GEMM sweep
over M and split counts, the pooler + RMSNorm + NVFP4 and the o_proj + dual
norm, each as µs per call over >= 200 calls with 48 rotated weight copies),
the CPU oracle on a bounded sample, and the SM clocks sampled during the timed
region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun) each rank runs an independent replica on its own GPU
(the path has no exchange step); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "skinny-GEMM(+fused epilogue) achieved HBM GB/s and % of GB300 peak, µs/call, M=1..16"
FALLBACK_HBM_GBS = 6800.0
M_ROWS = 16
LAYERS = 48
WORKLOAD = ("decode chain, 48 layers, M=16: o_proj GEMM [8192,8192] + dual norm -> pooler GEMM "
            "[4096,8192] + RMSNorm + NVFP4 -> unpooler GEMM [8192,4096]")
GEMM_SOURCES = ["nvfp4_sm_skinny_gb300/csrc/sk_kernels.cu", "nvfp4_sm_skinny_gb300/csrc/sk_ptx.cuh",
                "nvfp4_sm_skinny_gb300/csrc/sk_internal.h", "nvfp4_sm_skinny_gb300/csrc/sk_api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "skinny_gemm_chain_m16.md")
# Reference / CPU-baseline sample: 1/64 of each GEMM's output features (all of
# K) plus the two epilogues on full rows, M = 16.
SAMPLE_FRACTION = 64


# ------------------------------------------------------------ distributed ----
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a group)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(bytes_per_rank_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job GB/s: bytes all ranks processed over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / max_seconds / 1e9


# ------------------------------------------------------------------ peaks ----
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in d and isinstance(d[key], (int, float)):
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM bytes of the GEMM kernel from the committed ncu summary,
    or None if absent or taken on different kernel sources."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    mh = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    mt = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != gemm_source_hash():
        return None
    return float(mt.group(1))


# ----------------------------------------------------------------- clocks ----
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id, self.proc, self.out = bus_id, None, None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.bus_id:
            cmd[1:1] = ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def bus_id_of(device_index: int):
    import torch

    p = torch.cuda.get_device_properties(device_index)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return None


# ------------------------------------------------------ oracle (CPU) arm ----
class OracleSample:
    """A bounded slice of one chain layer computed by the CPU oracle: 1/64 of
    each GEMM's output features over all of K, and both epilogues on full
    rows, at M = 16. Weights are seeded on the CPU (same distributions as the
    chain)."""

    def __init__(self):
        import numpy as np

        import oracle
        from nvfp4_sm_skinny_gb300 import synth

        oracle.build()
        self.oracle, self.np = oracle, np
        H, P, m, f = synth.HIDDEN, synth.POOLED, M_ROWS, SAMPLE_FRACTION
        b = synth.bits
        self.x = b(synth.normal_bf16((m, H), 1.0, 0))
        self.w_o = b(synth.normal_bf16((H // f, H), 0.02, 10000))
        self.w_p = b(synth.normal_bf16((P // f, H), 0.02, 10001))
        self.w_u = b(synth.normal_bf16((H // f, P), 0.02, 10002))
        self.post_w = b(synth.normal_bf16((H,), 0.1, 10003, mean=1.0))
        self.pre_w = b(synth.normal_bf16((H,), 0.1, 10004, mean=1.0))
        self.beta = b(synth.uniform_bf16((H,), 0.5, 1.5, 10005))
        self.norm_w = b(synth.normal_bf16((P,), 0.1, 10006))
        self.s = synth.normal_f32((m, H), 503).numpy()
        self.partial = np.tile(b(synth.normal_bf16((m, H // f), 1.0, 7)), (1, f))
        self.y = np.tile(b(synth.normal_bf16((m, P // f), 1.0, 8)), (1, f))
        self.z_in = b(synth.normal_bf16((m, P), 1.0, 9))
        self.bytes = (2 * (H // f) * H + 2 * m * H + 2 * m * (H // f)) + \
                     (2 * (P // f) * H + 2 * m * H + 2 * m * (P // f)) + \
                     (2 * (H // f) * P + 2 * m * P + 2 * m * (H // f)) + \
                     (3 * 2 * H + 2 * 4 * m * H + 2 * m * H) + \
                     (2 * P + 4 + m * P // 2 + m * P // 16 + 2 * m * P)

    def step(self):
        o = self.oracle
        f = SAMPLE_FRACTION
        p_slice = o.gemm_bf16(self.x, self.w_o)
        self.partial[:, : p_slice.shape[1]] = p_slice
        s, u = o.dual_norm(self.partial, self.s, self.post_w, 1.0, self.beta, self.pre_w, 1e-6, 1e-6)
        y_slice = o.gemm_bf16(u, self.w_p)
        self.y[:, : y_slice.shape[1]] = y_slice
        a, a_sf, z = o.rmsnorm_nvfp4(self.y, self.norm_w, 1e-6, 1.0, 448.0)
        o.gemm_bf16(z, self.w_u)
        _ = f


def cpu_baseline(seconds: float = 12.0):
    smp = OracleSample()
    smp.step()                     # warm caches, build
    t0 = time.perf_counter()
    n = 0
    while True:
        smp.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": round(smp.bytes * n / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} oracle steps of a 1/{SAMPLE_FRACTION} slice of one chain layer (each GEMM's "
                      f"output features over all of K, both epilogues on full rows), M=16, single thread, "
                      f"{el:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    smp = OracleSample()
    for _ in range(args.warmup):
        smp.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.step()
    el = time.perf_counter() - t0
    value = smp.bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"1/{SAMPLE_FRACTION} slice of one layer per step",
                   "m": M_ROWS},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step a 1/{SAMPLE_FRACTION} slice of one chain layer, M=16"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU arm ----
def time_graph(graph, steps: int, stream) -> float:
    """Seconds for `steps` replays, CUDA events on the replay stream."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def time_graph_steps(graph, steps: int, stream):
    """(total seconds, per-replay seconds) for `steps` back-to-back replays:
    one CUDA event between consecutive replays on the replay stream."""
    import torch

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            graph.replay()
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(steps)]
    return ev[0].elapsed_time(ev[-1]) / 1e3, per


def quantiles(xs, qs=(0.1, 0.5, 0.9)):
    """Linear-interpolated quantiles of a non-empty list."""
    v = sorted(xs)
    out = []
    for q in qs:
        pos = q * (len(v) - 1)
        lo = int(pos)
        hi = min(lo + 1, len(v) - 1)
        out.append(v[lo] + (v[hi] - v[lo]) * (pos - lo))
    return out


def single_call_workloads(sk, synth, dev, stream, peak, min_calls: int = 200, copies: int = 48,
                          only: str | None = None):
    """Per-call timings of the single-call workloads, each point a CUDA graph of
    one call per weight copy (48 copies, more bytes than L2), replayed until at
    least `min_calls` calls are timed: µs per call as median, p10 and p90 over
    the replays, algorithmic GB/s and % of the HBM peak at the median.

    * the unpooler shard M=1 [1024,4096] and the GEMM sweep M in {1,2,4,8,16} x
      (N,K) in {(1024,4096),(8192,4096)} at the automatic split, plus every
      split count S in {1,2,4,8} at M=16;
    * the pooler GEMM [4096,8192] + RMSNorm + NVFP4 at b in {1,8,16};
    * the o_proj GEMM [8192,1024] + dual norm at b in {1,4,16};
    * the weight-only NVFP4 GEMM at M in {1,16} on [8192,8192], [4096,8192]
      and [8192,4096] (bytes: codes, scales, activations and output).
    Automatic-split points also report `hinted_us_p50`: the same calls, each
    told the next call's weight (sk_gemm_prefetch_next); GEMM points also
    `x_ready_us_p50`: hinted calls on an input no kernel writes
    (sk_gemm_bf16_ex, SK_GEMM_X_READY), which overlap call with call. `only`
    (a substring of the point names) restricts the run to matching points."""
    import torch

    bf = dict(dtype=torch.bfloat16, device=dev)
    out = {}

    def timed(calls):
        with torch.cuda.stream(stream):
            for c in calls:
                c()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
        for _ in range(3):
            with torch.cuda.stream(stream):
                g.replay()
        reps = max(5, -(-min_calls // len(calls)))
        _, per = time_graph_steps(g, reps, stream)
        del g
        return [t / len(calls) for t in per], reps * len(calls)

    def hinted(ws, call):
        def one(i):
            def f():
                sk.gemm_prefetch_next(ws[(i + 1) % len(ws)])
                call(ws[i])
            return f
        return [one(i) for i in range(len(ws))]

    def want(key):
        return only is None or only in key

    def put(key, workload, m, n, k, splits, nbytes, per, ncalls, hint_per=None, xr_per=None):
        p10, p50, p90 = quantiles(per)
        gbs = nbytes / p50 / 1e9
        r = {"workload": workload, "m": m, "n": n, "k": k, "splits": splits,
             "us_p50": round(p50 * 1e6, 3), "us_p10": round(p10 * 1e6, 3),
             "us_p90": round(p90 * 1e6, 3), "calls": ncalls, "bytes": nbytes,
             "gbs": round(gbs, 1), "pct_of_peak": round(100.0 * gbs / peak, 2)}
        if hint_per is not None:
            h50 = quantiles(hint_per, (0.5,))[0]
            r["hinted_us_p50"] = round(h50 * 1e6, 3)
            r["hinted_pct_of_peak"] = round(100.0 * nbytes / h50 / 1e9 / peak, 2)
        if xr_per is not None:
            x50 = quantiles(xr_per, (0.5,))[0]
            r["x_ready_us_p50"] = round(x50 * 1e6, 3)
            r["x_ready_pct_of_peak"] = round(100.0 * nbytes / x50 / 1e9 / peak, 2)
        out[key] = r

    for n, k in ((1024, 4096), (8192, 4096)):
        if not any(want(f"gemm_m{m}_n{n}_k{k}") for m in (1, 2, 4, 8, 16)):
            continue
        ws = [synth.gemm_weight(n, k, i, device=dev) for i in range(copies)]
        for m in (1, 2, 4, 8, 16):
            if not want(f"gemm_m{m}_n{n}_k{k}"):
                continue
            x = synth.gemm_x(m, k).to(dev)
            y = torch.empty(m, n, **bf)
            nbytes = 2 * n * k + 2 * m * k + 2 * m * n
            per, nc = timed([lambda w=w: sk.gemm_bf16(x, w, out=y, stream=stream) for w in ws])
            hper, _ = timed(hinted(ws, lambda w: sk.gemm_bf16(x, w, out=y, stream=stream)))
            # x is written by no kernel here (one host copy, synchronised): the
            # calls may read it without waiting for the call ahead of them
            torch.cuda.synchronize(dev)
            xper, _ = timed(hinted(ws, lambda w: sk.gemm_bf16(x, w, out=y, stream=stream,
                                                              x_ready=True)))
            wl = "unpooler GEMM" if m == 1 and n == 1024 else "GEMM"
            put(f"gemm_m{m}_n{n}_k{k}", wl, m, n, k, f"auto({sk.gemm_splits(m, n, k)})", nbytes,
                per, nc, hper, xper)
            if m == 16:
                for S in (1, 2, 4, 8):
                    if sk.gemm_supported(m, n, k, S) is not None:
                        continue
                    per, nc = timed([lambda w=w, S=S: sk.gemm_bf16(x, w, out=y, splits=S,
                                                                  stream=stream) for w in ws])
                    put(f"gemm_m{m}_n{n}_k{k}_s{S}", "GEMM", m, n, k, S, nbytes, per, nc)
        sk.gemm_prefetch_next(None)
        del ws
        torch.cuda.empty_cache()

    H, P = synth.HIDDEN, synth.POOLED
    pool_b = [b for b in (1, 8, 16) if want(f"pooler_nvfp4_b{b}")]
    ws = [synth.normal_bf16((P, H), 0.02, 200 + i, device=dev) for i in range(copies)] if pool_b else []
    nw = synth.normal_bf16((P,), 0.1, 300, device=dev)
    gs = torch.tensor([300.0], dtype=torch.float32, device=dev)
    for b in pool_b:
        x = synth.normal_bf16((b, H), 1.0, 0, device=dev)
        a = torch.empty(b, P // 2, dtype=torch.uint8, device=dev)
        a_sf = torch.empty(b, P // 16, dtype=torch.uint8, device=dev)
        wsp = torch.empty(sk.gemm_rmsnorm_nvfp4_workspace(b, P), dtype=torch.uint8, device=dev)

        def call(w, x=x, a=a, a_sf=a_sf, wsp=wsp):
            sk.gemm_rmsnorm_nvfp4(x, w, nw, synth.EPS, synth.GAIN_CENTER, gs, a=a, a_sf=a_sf,
                                  workspace=wsp, stream=stream)
        per, nc = timed([lambda w=w: call(w) for w in ws])
        hper, _ = timed(hinted(ws, call))
        put(f"pooler_nvfp4_b{b}", "pooler GEMM + RMSNorm + NVFP4", b, P, H,
            f"auto({sk.gemm_splits(b, P, H)})",
            2 * P * H + 2 * b * H + 2 * P + 4 + b * P // 2 + b * P // 16, per, nc, hper)
    sk.gemm_prefetch_next(None)
    del ws
    torch.cuda.empty_cache()

    K = synth.OPROJ_K
    dual_b = [b for b in (1, 4, 16) if want(f"oproj_dual_b{b}")]
    ws = [synth.normal_bf16((H, K), 0.02, 400 + i, device=dev) for i in range(copies)] if dual_b else []
    post_w = synth.normal_bf16((H,), 0.1, 500, mean=1.0, device=dev)
    pre_w = synth.normal_bf16((H,), 0.1, 501, mean=1.0, device=dev)
    beta = synth.uniform_bf16((H,), 0.5, 1.5, 502, device=dev)
    for b in dual_b:
        x = synth.normal_bf16((b, K), 1.0, 0, device=dev)
        # the residual stream is updated in place and drifts from call to call
        s_res = synth.normal_f32((b, H), 503, device=dev)
        o = torch.empty(b, H, **bf)
        wsp = torch.empty(sk.gemm_dual_norm_workspace(b, H), dtype=torch.uint8, device=dev)

        def call(w, x=x, s_res=s_res, o=o, wsp=wsp):
            sk.gemm_dual_norm(x, w, s_res, post_w, 1.0, beta, pre_w, out=o, eps_post=synth.EPS,
                              eps_pre=synth.EPS, workspace=wsp, stream=stream)
        per, nc = timed([lambda w=w: call(w) for w in ws])
        hper, _ = timed(hinted(ws, call))
        put(f"oproj_dual_b{b}", "o_proj GEMM + dual norm", b, H, K,
            f"auto({sk.gemm_splits(b, H, K)})",
            2 * H * K + 2 * b * K + 3 * 2 * H + 2 * 4 * b * H + 2 * b * H, per, nc, hper)
    sk.gemm_prefetch_next(None)
    del ws
    torch.cuda.empty_cache()

    # weight-only NVFP4 GEMM: BF16 weights ~ N(0, 0.02) quantized on the device
    # (sk_nvfp4_quantize, gs = 448 * 6 / amax), 4.5 bits per weight
    for n, k in ((8192, 8192), (4096, 8192), (8192, 4096)):
        if not any(want(f"nvfp4w_m{m}_n{n}_k{k}") for m in (1, 16)):
            continue
        wqs, wsfs, wss = [], [], []
        for i in range(copies):
            w = synth.normal_bf16((n, k), 0.02, 600 + i, device=dev)
            gs_i = (2688.0 / w.float().abs().amax().clamp_min(1e-30)).reshape(1)
            wq, wsf = sk.nvfp4_quantize(w, gs_i, stream=None)
            wqs.append(wq)
            wsfs.append(wsf)
            wss.append((1.0 / gs_i).contiguous())
            del w
        torch.cuda.synchronize(dev)
        for m in (1, 16):
            if not want(f"nvfp4w_m{m}_n{n}_k{k}"):
                continue
            x = synth.gemm_x(m, k).to(dev)
            y = torch.empty(m, n, **bf)
            per, nc = timed([lambda i=i: sk.gemm_nvfp4w(x, wqs[i], wsfs[i], wss[i], out=y, stream=stream)
                             for i in range(copies)])
            put(f"nvfp4w_m{m}_n{n}_k{k}", "weight-only NVFP4 GEMM", m, n, k,
                f"auto({sk.gemm_nvfp4w_splits(m, n, k)})",
                n * k // 2 + n * k // 16 + 4 + 2 * m * k + 2 * m * n, per, nc)
        del wqs, wsfs, wss
        torch.cuda.empty_cache()
    return out


def run_gpu(args, world, rank, local):
    import torch

    from __graft_entry__ import build
    build()
    import nvfp4_sm_skinny_gb300 as sk
    from nvfp4_sm_skinny_gb300 import synth
    from nvfp4_sm_skinny_gb300.chain import DecodeChain, gemm_bytes, layer_bytes

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    L = args.layers
    chain = DecodeChain(L, M_ROWS, dev)
    h0 = synth.normal_bf16((M_ROWS, synth.HIDDEN), 1.0, 0).to(dev)
    s0 = synth.normal_f32((M_ROWS, synth.HIDDEN), 503).to(dev)
    chain.calibrate(synth.normal_bf16((M_ROWS, synth.HIDDEN), 1.0, 1000).to(dev), s0)
    chain.set_input(h0, s0)
    g_chain = chain.capture(chain.forward)
    g_gemm = chain.capture(chain.gemms_only)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    assert sk.device_status() == 0

    bytes_step = layer_bytes(M_ROWS)["total"] * L
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            g_chain.replay()
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps of the whole chain
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(bus_id_of(local) if rank == 0 else None)
    if rank == 0:
        sampler.start()
        time.sleep(0.25)
    t_chain, step_s = time_graph_steps(g_chain, args.steps, stream)
    clocks = sampler.stop() if rank == 0 else None
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t_max = reduce_max(t_chain, dist, dev)
    value = aggregate_rate(bytes_step, args.steps, world, t_max)

    # ---- the dominant kernel alone: the chain's GEMM launches
    for _ in range(max(3, args.warmup // 2)):
        with torch.cuda.stream(stream):
            g_gemm.replay()
    gemm_steps = max(10, args.steps // 2)
    t_gemm = time_graph(g_gemm, gemm_steps, stream)
    launches = L * DecodeChain.gemm_launches_per_layer
    per_launch_s = t_gemm / (gemm_steps * launches)
    gemm_bytes_launch = gemm_bytes(M_ROWS) / DecodeChain.gemm_launches_per_layer
    achieved = gemm_bytes_launch / per_launch_s / 1e9
    peak, peak_src = hbm_peak()
    traffic = recorded_traffic()

    # ---- per-op µs/call inside the chain's launch configuration
    per_op = {}
    lb = layer_bytes(M_ROWS)
    for name, fn in (("oproj_dual", lambda: [chain.layer_op(l, 0) for l in range(L)]),
                     ("pooler_nvfp4", lambda: [chain.layer_op(l, 1) for l in range(L)]),
                     ("unpooler", lambda: [chain.layer_op(l, 2) for l in range(L)])):
        g = chain.capture(fn)
        for _ in range(3):
            with torch.cuda.stream(stream):
                g.replay()
        reps = max(5, args.steps // 4)
        t = time_graph(g, reps, stream)
        us = t / (reps * L) * 1e6
        per_op[name] = {"us_per_call": round(us, 3),
                        "gbs": round(lb[name] / (us * 1e-6) / 1e9, 1)}
        del g

    # ---- end to end through the C-ABI calls with host buffers
    pin = dict(pin_memory=True)
    h_host = h0.cpu().pin_memory()
    s_host = s0.cpu().pin_memory()
    # Two buffer sets on the same weights, one graph each, so that step i + 1's
    # inputs are copied in and step i - 1's results copied out while step i
    # runs, as a serving loop overlaps its I/O with compute; each set has its
    # own pinned result buffers, read on the host while the next step runs.
    chain_b = chain.twin()
    chain_b.set_input(h0, s0)
    g_chain_b = chain_b.capture(chain_b.forward)
    sets = [(chain, g_chain), (chain_b, g_chain_b)]
    outs = [(torch.empty(M_ROWS, synth.HIDDEN, dtype=torch.bfloat16, **pin),
             torch.empty(M_ROWS, synth.POOLED // 2, dtype=torch.uint8, **pin),
             torch.empty(M_ROWS, synth.POOLED // 16, dtype=torch.uint8, **pin)) for _ in range(2)]
    h2d = h_host.numel() * 2 + s_host.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs[0])
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_steps_run(n_steps):
        """n_steps decode steps as a pipelined serving loop runs them. Step i
        uses buffer set i % 2: its inputs are copied in on s_in once step
        i - 2's graph and result copies on that set are done, its graph runs on
        the compute stream once they have landed, and its results are copied
        out on s_out once it has run. The host queues step i + 1 before it
        waits for step i's results."""
        out_done = [None, None]
        for i in range(n_steps):
            k = i % 2
            c, g = sets[k]
            out_h, out_a, out_sf = outs[k]
            with torch.cuda.stream(s_in):
                if out_done[k] is not None:
                    s_in.wait_event(out_done[k])
                c.h[0].copy_(h_host, non_blocking=True)
                c.s.copy_(s_host, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in)
                g.replay()
                ev_g = torch.cuda.Event()
                ev_g.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_g)
                out_h.copy_(c.h[L], non_blocking=True)
                out_a.copy_(c.a[L - 1], non_blocking=True)
                out_sf.copy_(c.a_sf[L - 1], non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
            out_done[k] = ev_o
            if i >= 1:
                out_done[(i - 1) % 2].synchronize()  # step i - 1's results are on the host
        out_done[(n_steps - 1) % 2].synchronize()

    e2e_steps_run(3)
    e2e_steps = max(10, min(args.steps, 300))
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_steps_run(e2e_steps)
    t_e2e = reduce_max(time.perf_counter() - t0, dist, dev)
    e2e_value = aggregate_rate(bytes_step, e2e_steps, world, t_e2e)
    # both buffer sets ran the same inputs: their results must agree bit for bit
    if not all(torch.equal(a.view(torch.uint8), b.view(torch.uint8)) for a, b in zip(*outs)):
        raise RuntimeError("the two buffer sets of the end-to-end loop disagree")
    del g_chain_b, chain_b
    status = sk.device_status()

    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = single_call_workloads(sk, synth, dev, stream, peak)
        status |= sk.device_status()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(t_max / args.steps * 1e3, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) weights per layer, N(0,1) activations)",
            "config": {"workload": WORKLOAD if L == LAYERS else WORKLOAD.replace("48 layers", f"{L} layers"),
                       "m": M_ROWS, "layers": L,
                       "weights_bytes": L * (2 * 8192 * 8192 + 2 * 2 * 4096 * 8192),
                       "l2": f"inputs larger than L2 ({L * 256} MiB of weights per step), no flush",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "bytes_per_step": bytes_step},
            "pct_of_peak": round(100.0 * value / world / peak, 2),
            "step_ms": dict(zip(("p10", "p50", "p90"),
                                (round(q * 1e3, 4) for q in quantiles(step_s)))),
            "peak_hbm_gbs": {"value": peak, "source": peak_src},
            "per_op": per_op,
            "per_config": per_config,
            "roofline": {"bound": "hbm", "kernel": "sk::gemm_kernel (all chain GEMM launches)",
                         "achieved": round(achieved, 2), "peak": peak,
                         "peak_source": f"{peak_src} HBM copy bandwidth", "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": round(gemm_bytes_launch),
                         "launch_us": round(per_launch_s * 1e6, 3)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * L * DecodeChain.launches_per_layer,
            "clocks": clocks,
            "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- sweep ----
def run_sweep(args, local):
    """The single-call workloads of the default run's per_config, alone: one
    JSON line per point, then a markdown table. --only restricts the points
    (a substring of their names, e.g. nvfp4w_m16_n8192_k8192)."""
    import torch

    from __graft_entry__ import build
    build()
    import nvfp4_sm_skinny_gb300 as sk
    from nvfp4_sm_skinny_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peak, peak_src = hbm_peak()
    stream = torch.cuda.Stream(dev)
    rows = single_call_workloads(sk, synth, dev, stream, peak, only=args.only)
    for key, r in rows.items():
        print(json.dumps(dict(point=key, **r)), flush=True)
    print(f"\n| point | workload | M | N | K | splits | µs/call p50 (p10-p90) | GB/s | % of {peak_src} "
          f"peak ({peak:.0f} GB/s) | hinted µs | x ready µs |")
    print("|---|---|---|---|---|---|---|---|---|---|---|")
    for key, r in rows.items():
        print(f"| {key} | {r['workload']} | {r['m']} | {r['n']} | {r['k']} | {r['splits']} | "
              f"{r['us_p50']:.2f} ({r['us_p10']:.2f}-{r['us_p90']:.2f}) | {r['gbs']:.0f} | "
              f"{r['pct_of_peak']:.1f} | {r.get('hinted_us_p50', '')} | {r.get('x_ready_us_p50', '')} |")
    print(f"\ndevice status {sk.device_status()}")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["sk", "reference"], default="sk")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the single-call workloads (per_config) after the chain")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="chain depth (48 is the benchmark; fewer only for small profiling runs)")
    ap.add_argument("--sweep", action="store_true",
                    help="per-call timings of the single-call workloads instead of the chain")
    ap.add_argument("--only", default=None,
                    help="with --sweep: only the points whose names contain this string")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.sweep:
        return run_sweep(args, local)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
