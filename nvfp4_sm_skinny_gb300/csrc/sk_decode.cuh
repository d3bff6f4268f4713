// Fused decode layer: the o_proj GEMM, the attention-boundary dual norm, the
// pooler GEMM with the pre-expert RMSNorm and NVFP4, and the unpooler GEMM in
// one persistent kernel (one CTA per SM, all resident: a cooperative launch).
//
// Why one kernel: each step of the layer streams a weight from HBM, and the
// weights never depend on the activations. A single producer thread per CTA
// therefore streams the three weights back to back through one shared-memory
// ring while the rest of the CTA waits for the activations of each GEMM; the
// norms, the NVFP4 quantization and the grid-wide syncs between the steps run
// while the ring keeps filling. Separate kernels would drain and refill the
// memory pipeline at every boundary.
//
// Roles (kDecThreads threads): warp 0 lane 0 issues the TMA copies (weights
// as soon as a ring slot is free; activations once the step's input is
// complete), lane 0 of warps 1..kDecIssuers issue the tcgen05 MMAs (box j of a
// stage to issuer j mod kDecIssuers, each with its own accumulators), and the
// last four warps (one per TMEM lane quadrant) run the epilogues: dual norm,
// RMSNorm + NVFP4, stores. The arithmetic of each
// epilogue matches the standalone kernels (same FP32 operations per element;
// reductions in a fixed order), so results are bitwise reproducible run to run.
//
// Included into sk_kernels.cu (it shares the device status word).

namespace sk {

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned *p) {
  return *reinterpret_cast<const volatile unsigned *>(p);
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ float bf16_round_f32(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Sum of v[t] over the 128 epilogue threads, for each of 16 tokens, in a fixed
// order (shuffle-down tree in each warp, then the four warps in order). The
// result lands in tot[0..15] (shared), visible to every epilogue thread.
__device__ __forceinline__ void epi_sum16(const float (&v)[16], float *red, float *tot, int ew,
                                          int lane) {
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    float x = v[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
    if (lane == 0) red[ew * 16 + t] = x;
  }
  epi_bar();
  const int e = ew * 32 + lane;
  if (e < 16) tot[e] = ((red[e] + red[16 + e]) + red[32 + e]) + red[48 + e];
  epi_bar();
}

// Sum over the CTAs of the grid of part[c][t] (global, written before the last
// grid barrier), in CTA order in eight fixed chunks, for each of 16 tokens;
// every CTA computes the same bits. Result in tot[0..15].
__device__ __forceinline__ void epi_grid_sum16(const float *part, int G, float *tot, int ew,
                                               int lane) {
  const int e = ew * 32 + lane;
  const int t = e >> 3, j = e & 7;
  const int chunk = (G + 7) / 8;
  const int c0 = j * chunk, c1 = min(G, c0 + chunk);
  float acc = 0.0f;
  bool first = true;
  // all loads of a batch are issued before the first add: one L2 round trip
  // per batch instead of one per CTA
  constexpr int kBatch = 24;
  for (int cb = c0; cb < c1; cb += kBatch) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) v[u] = cb + u < c1 ? __ldcg(part + (cb + u) * 16 + t) : 0.0f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (cb + u < c1) {
        acc = first ? v[u] : acc + v[u];
        first = false;
      }
    }
  }
  // the eight chunk sums of token t sit in eight consecutive lanes
  float total = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float v = __shfl_sync(0xffffffffu, acc, (lane & ~7) + q);
    total = q == 0 ? v : total + v;
  }
  if (j == 0) tot[t] = total;
  epi_bar();
}

// Grid-wide barrier among the epilogue warps of all CTAs: arrive on the
// counter, wait (bounded, backing off between polls) until it reaches
// `target`. Only thread 0 of the epilogue touches global memory here. On
// success it raises `ready_flag` (shared, may be null) for the producer; on
// timeout or abort it raises the CTA's abort flag. Returns false on failure.
__device__ __forceinline__ bool epi_grid_sync(unsigned *bar, unsigned target, unsigned *gabort,
                                              int e, volatile uint32_t *ready_flag,
                                              volatile uint32_t *abort_flag) {
  __shared__ int ok_s;
  epi_bar();
  if (e == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_u32(bar) < target) {
      __nanosleep(32);
      if (*abort_flag || ld_volatile_u32(gabort)) {
        ok = 0;
        break;
      }
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_GRID);
        atomicExch(gabort, 1u);
        ok = 0;
        break;
      }
    }
    // the acquire load that saw the final count orders this CTA's later reads
    // after every CTA's release (fence + add) of its partials
    if (ok && ready_flag) *ready_flag = 1;
    if (!ok) *abort_flag = 1;
    ok_s = ok;
  }
  epi_bar();
  return ok_s != 0;
}

// Bounded wait of the producer / MMA threads on a ring barrier. Polls only
// shared memory; the grid-wide abort word is read once a wait has lasted long.
__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                         const unsigned *gabort, uint32_t status_bit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if ((++spins & 255) == 0) {
      const uint64_t dt = globaltimer_ns() - t0;
      if (dt > 100000ull && ld_volatile_u32(gabort)) {
        *abort_flag = 1;
        return false;
      }
      if (dt > kWaitLimitNs) {
        atomicOr(&g_device_status, status_bit);
        atomicExch(const_cast<unsigned *>(gabort), 1u);
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_layer_kernel(const __grid_constant__ DecodeMaps maps, const DecodeArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int B = args.bps;
  const int S = args.stages;
  const int slot_w = args.slot_w;
  const DecodeLayout lay = decode_layout(slot_w, S, B);
  uint8_t *s_w = smem;
  uint8_t *s_x = smem + lay.x_off;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + kDecPhases);
  volatile uint32_t *abort_flag = tmem_slot + 1;
  volatile uint32_t *x_ready = tmem_slot + 2;  // [1], [2]: inputs of the pooler / unpooler complete
  float *red = reinterpret_cast<float *>(smem + lay.red_off);
  float *tot = red + 64;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + S);
  const uint32_t done0 = smem_u32(bars + 2 * S);

  // stage sequence of this CTA: the phases it has a tile in, in order
  int nst[kDecPhases], st0[kDecPhases], total = 0;
#pragma unroll
  for (int p = 0; p < kDecPhases; ++p) {
    nst[p] = c < args.tiles[p] ? (args.nkb[p] + B - 1) / B : 0;
    st0[p] = total;
    total += nst[p];
  }
  // first 64-wide K block of stage ls of phase p
  auto kb_of = [&](int ls, int /*p*/) { return ls * B; };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 2);  // the weight arrival and the activation arrival
      mbar_init(empty0 + 8 * s, kDecIssuers);
    }
    for (int p = 0; p < kDecPhases; ++p) mbar_init(done0 + 8 * p, kDecIssuers);
    *abort_flag = 0;
    x_ready[0] = 0;
    x_ready[1] = 0;
    fence_barrier_init();
    for (int p = 0; p < kDecPhases; ++p) {
      tma_prefetch_map(&maps.w[p]);
      tma_prefetch_map(&maps.x[p]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kDecTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      bool ready[kDecPhases] = {false, false, false};
      int xi = 0;  // stages below xi have their activation copies issued
      auto phase_of = [&](int i) {
        int p = 0;
        while (p + 1 < kDecPhases && i >= st0[p + 1]) ++p;
        return p;
      };
      // activation copies of armed stages whose input is complete
      auto issue_x = [&](int armed) {
        while (xi < armed) {
          const int p = phase_of(xi);
          if (!ready[p]) {
            // set by this CTA's epilogue once the grid barrier before step p passed
            if (p == 0 || !x_ready[p - 1]) break;
            fence_proxy_async_global();  // generic-proxy stores of other CTAs -> TMA reads
            ready[p] = true;
          }
          const int s = xi % S;
          mbar_arrive_expect_tx(full0 + 8 * s, B * kSlotXBytes);
          tma_load_3d(smem_u32(s_x + s * B * kSlotXBytes), &maps.x[p], full0 + 8 * s, 0, 0,
                      kb_of(xi - st0[p], p), pol_x);
          ++xi;
        }
      };
      auto arm_w = [&](int i) {
        const int p = phase_of(i), s = i % S;
        // one copy: B blocks of h[p] rows (blocks past K arrive as zeros)
        mbar_arrive_expect_tx(full0 + 8 * s, B * args.h[p] * 128);
        tma_load_3d(smem_u32(s_w + s * B * slot_w), &maps.w[p], full0 + 8 * s, 0, c * args.h[p],
                    kb_of(i - st0[p], p), pol_w);
      };
      const int fill = total < S ? total : S;
      for (int i = 0; i < fill; ++i) arm_w(i);  // weights first: never written by a kernel
      griddep_wait();                           // h_in is written by the previous kernel
      ready[0] = true;
      issue_x(fill);
      bool ok = true;
      for (int i = fill; i < total && ok; ++i) {
        const int s = i % S;
        const uint32_t par = ((i / S) & 1) ^ 1;
        const uint64_t t0 = globaltimer_ns();
        uint32_t spins = 0;
        while (!mbar_try_wait(empty0 + 8 * s, par)) {
          issue_x(i);  // keep activations flowing while the ring is full
          if (*abort_flag) { ok = false; break; }
          if ((++spins & 255) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_device_status, SK_DEVICE_WAIT_PRODUCER);
            atomicExch(args.gabort, 1u);
            *abort_flag = 1;
            ok = false;
            break;
          }
        }
        if (!ok) break;
        arm_w(i);
        issue_x(i + 1);
      }
      // the last activations wait for their step's input
      const uint64_t t0 = globaltimer_ns();
      while (ok && xi < total) {
        issue_x(total);
        if (xi >= total || *abort_flag) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(&g_device_status, SK_DEVICE_WAIT_PRODUCER);
          atomicExch(args.gabort, 1u);
          *abort_flag = 1;
          break;
        }
        __nanosleep(128);
      }
    }
  } else if (warp <= kDecIssuers) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuers
      const int q = warp - 1;
      int i = 0;
      bool ok = true;
      for (int p = 0; p < kDecPhases && ok; ++p) {
        if (nst[p] == 0) continue;
        bool started = false;  // this issuer's accumulators hold this phase's partial sum
        for (int ls = 0; ls < nst[p]; ++ls, ++i) {
          const int s = i % S;
          const uint32_t par = (i / S) & 1;
          if (!dec_wait(full0 + 8 * s, par, abort_flag, args.gabort, SK_DEVICE_WAIT_MMA)) ok = false;
          if (!ok) break;
          tc_fence_after_sync();
          const int nb = min(B, args.nkb[p] - kb_of(ls, p));
          for (int j = q; j < nb; j += kDecIssuers) {
            // block j of the stage: h[p] rows of 128 bytes after block j - 1
            const uint64_t adesc = smem_desc_k128(smem_u32(s_w + s * B * slot_w + j * args.h[p] * 128));
            const uint64_t bdesc = smem_desc_k128(smem_u32(s_x + (s * B + j) * kSlotXBytes));
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk)
              tc_mma_bf16(tmem + static_cast<uint32_t>(acc_index(q, kk) * kTokTile), adesc + 2 * kk,
                          bdesc + 2 * kk, kIdesc, started || kk > 0);
            started = true;
          }
          tc_commit(empty0 + 8 * s);
        }
        tc_commit(done0 + 8 * p);
      }
      if (!ok) {
        for (int p = 0; p < kDecPhases; ++p) tc_commit(done0 + 8 * p);
      }
    }
  } else {
    // -------------------------------------------------------- epilogue
    const int ew = warp - 1 - kDecIssuers;        // 0..3
    const int e = ((warp & 3) << 5) + lane;       // TMEM lane = tile row
    const int m = args.m, H = args.H, P = args.P;
    const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float v[16];
    bool ok = true;

    // ---- o_proj + dual norm
    const int h0 = args.h[0];
    const int n = c * h0 + e;
    const bool has0 = c < args.tiles[0];
    const bool valid0 = has0 && e < h0 && n < H;
    float w1v = 1.0f, bv = 0.0f, w2v = 0.0f, sv[16];
    if (valid0) {
      if (args.post_w) w1v = __fadd_rn(bf16_bits_to_f32(args.post_w[n]), args.gc_post);
      bv = bf16_bits_to_f32(args.beta[n]);
      w2v = __fadd_rn(bf16_bits_to_f32(args.pre_w[n]), args.gc_pre);
    }
    griddep_wait();  // the residual stream may be written by the previous kernel
#pragma unroll
    for (int t = 0; t < 16; ++t) sv[t] = (valid0 && t < m) ? args.s[static_cast<size_t>(t) * H + n] : 0.0f;
    float pv[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) pv[t] = 0.0f;
    if (has0) {
      if (!mbar_wait_idle(done0, 0, kWaitLimitNs)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
        atomicExch(args.gabort, 1u);
      }
      tc_fence_after_sync();
      tmem_sum_accumulators<kDecNumAcc>(taddr, acc_used(args.nkb[0], B, kDecIssuers), v);
      tc_fence_before_sync();
#pragma unroll
      for (int t = 0; t < 16; ++t) pv[t] = (valid0 && t < m) ? bf16_round_f32(v[t]) : 0.0f;
      if (args.p_out && valid0) {
        for (int t = 0; t < m; ++t)
          args.p_out[static_cast<size_t>(t) * H + n] = bf16_store_bits(pv[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t] = __fmul_rn(pv[t], pv[t]);
    epi_sum16(v, red, tot, ew, lane);
    if (e < 16) args.part[c * 16 + e] = tot[e];
    ok = epi_grid_sync(args.bar, 1u * G, args.gabort, e, nullptr, abort_flag);
    float r[16];
    if (ok) {
      epi_grid_sum16(args.part, G, tot, ew, lane);
#pragma unroll
      for (int t = 0; t < 16; ++t)
        r[t] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot[t], static_cast<float>(H)),
                                                     args.eps_post)));
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float q = __fmul_rn(__fmul_rn(pv[t], r[t]), w1v);
        sv[t] = __fmaf_rn(bv, q, __fmul_rn(args.alpha, sv[t]));
        if (valid0 && t < m) args.s[static_cast<size_t>(t) * H + n] = sv[t];
        v[t] = (valid0 && t < m) ? __fmul_rn(sv[t], sv[t]) : 0.0f;
      }
      epi_sum16(v, red, tot, ew, lane);
      if (e < 16) args.part[(G + c) * 16 + e] = tot[e];
      ok = epi_grid_sync(args.bar, 2u * G, args.gabort, e, nullptr, abort_flag);
    }
    if (ok) {
      epi_grid_sum16(args.part + G * 16, G, tot, ew, lane);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        r[t] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot[t], static_cast<float>(H)),
                                                     args.eps_pre)));
        if (valid0 && t < m)
          args.u[static_cast<size_t>(t) * H + n] = bf16_store_bits(__fmul_rn(__fmul_rn(sv[t], r[t]), w2v));
      }
      ok = epi_grid_sync(args.bar, 3u * G, args.gabort, e, &x_ready[0], abort_flag);
    }

    // ---- pooler + RMSNorm + NVFP4
    const int h1 = args.h[1];
    const int jrow = c * h1 + e;
    const bool has1 = c < args.tiles[1];
    const bool valid1 = has1 && e < h1 && jrow < P;
    float gv = 0.0f, yv[16];
    if (valid1) gv = __fadd_rn(bf16_bits_to_f32(args.norm_w[jrow]), args.gc_pool);
#pragma unroll
    for (int t = 0; t < 16; ++t) yv[t] = 0.0f;
    if (ok && has1) {
      if (!mbar_wait_idle(done0 + 8, 0, kWaitLimitNs)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
        atomicExch(args.gabort, 1u);
      }
      tc_fence_after_sync();
      tmem_sum_accumulators<kDecNumAcc>(taddr, acc_used(args.nkb[1], B, kDecIssuers), v);
      tc_fence_before_sync();
#pragma unroll
      for (int t = 0; t < 16; ++t) yv[t] = (valid1 && t < m) ? bf16_round_f32(v[t]) : 0.0f;
      if (args.y_out && valid1) {
        for (int t = 0; t < m; ++t)
          args.y_out[static_cast<size_t>(t) * P + jrow] = bf16_store_bits(yv[t]);
      }
    }
    if (ok) {
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = __fmul_rn(yv[t], yv[t]);
      epi_sum16(v, red, tot, ew, lane);
      if (e < 16) args.part[(2 * G + c) * 16 + e] = tot[e];
      ok = epi_grid_sync(args.bar, 4u * G, args.gabort, e, nullptr, abort_flag);
    }
    if (ok) {
      epi_grid_sum16(args.part + 2 * G * 16, G, tot, ew, lane);
      // the RMS factor of each token, once per CTA
      const int et = ew * 32 + lane;
      if (et < 16)
        tot[et] = __fdiv_rn(
            1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot[et], static_cast<float>(P)), args.eps_pool)));
      epi_bar();
      if (has1 && (e & ~31) < h1) {
        // rows of a 16-column NVFP4 block sit in 16 consecutive lanes (h1 is a
        // multiple of 16, so a block is wholly inside or outside the tile);
        // every lane of a warp that holds tile rows takes part in the shuffles.
        // Unrolled over the tokens so that independent tokens overlap.
        const float gs = *args.gs;
        const float inv_gs = __fdiv_rn(1.0f, gs);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (t >= m) break;
          const float rr = tot[t];
          const uint16_t zb = valid1 ? bf16_store_bits(__fmul_rn(__fmul_rn(yv[t], rr), gv)) : 0;
          const float zf = bf16_bits_to_f32(zb);
          float amax = fabsf(zf);
#pragma unroll
          for (int off = 8; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
          const float tq = __fmul_rn(__fdiv_rn(amax, 6.0f), gs);
          const uint32_t sf = cvt_f32_e4m3(tq);
          const float sff = cvt_e4m3_f32(sf);
          const float os = (sff == 0.0f) ? 0.0f : __fdiv_rn(1.0f, __fmul_rn(sff, inv_gs));
          const float vq = __fmul_rn(zf, os);
          const float vn = __shfl_xor_sync(0xffffffffu, vq, 1);
          if (valid1) {
            args.z[static_cast<size_t>(t) * P + jrow] = zb;
            if ((lane & 1) == 0)
              args.a[static_cast<size_t>(t) * (P / 2) + jrow / 2] =
                  static_cast<uint8_t>(cvt_f32x2_e2m1x2(vq, vn));
            if ((lane & 15) == 0)
              args.a_sf[static_cast<size_t>(t) * (P / 16) + jrow / 16] = static_cast<uint8_t>(sf);
          }
        }
      }
      ok = epi_grid_sync(args.bar, 5u * G, args.gabort, e, &x_ready[1], abort_flag);
    }

    // ---- unpooler
    const int h2 = args.h[2];
    const int n2 = c * h2 + e;
    const bool has2 = c < args.tiles[2];
    if (ok && has2) {
      if (!mbar_wait_idle(done0 + 16, 0, kWaitLimitNs)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
        atomicExch(args.gabort, 1u);
      }
      tc_fence_after_sync();
      tmem_sum_accumulators<kDecNumAcc>(taddr, acc_used(args.nkb[2], B, kDecIssuers), v);
      tc_fence_before_sync();
      if (e < h2 && n2 < H && !*abort_flag) {
#pragma unroll
        for (int t = 0; t < 16; ++t)
          if (t < m) args.h_out[static_cast<size_t>(t) * H + n2] = bf16_store_bits(v[t]);
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // after an abort some copies into the ring may still be in flight: give
    // them time to land before the CTA releases its shared memory
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kDecTmemCols);
}

cudaError_t launch_decode_layer(const DecodeMaps &maps, const DecodeArgs &args, int grid,
                                size_t smem, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeCooperative;
  attrs[na].val.cooperative = 1;
  ++na;
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel, maps, args);
}

size_t decode_smem_bytes(int slot_w, int stages, int bps) {
  return 1024 + static_cast<size_t>(decode_layout(slot_w, stages, bps).total);
}

}  // namespace sk
