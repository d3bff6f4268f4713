// Device code of libsk: the small-M skinny GEMM (TMA weight stream into a
// shared-memory ring, tcgen05 MMA into TMEM, cluster split-K reduced in DSMEM
// in a fixed order), the pre-expert RMSNorm + NVFP4 epilogue, the NVFP4
// quantizer and the attention-boundary dual norm.
//
// What the kernels compute follows the vLLM API pages of the Muse Spark
// specialized decode: cutedsl/gemm/unpooler (module docstring: the small-M
// product, the fixed-order split-K sum, -0.0 published as +0.0),
// cutedsl/moe/pooler_gather (module docstring: pre-expert norm and NVFP4
// layout; nvfp4_compute_output_scale and the cvt helpers), and
// cutedsl/oproj/batt (AttentionBoundary: the dual norm).
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "sk.h"
#include "sk_internal.h"
#include "sk_ptx.cuh"

namespace sk {

// OR of SK_DEVICE_WAIT_* bits, set by kernels whose bounded waits ran out.
__device__ uint32_t g_device_status;

constexpr uint32_t kIdesc = idesc_bf16_f32(kMmaM, kTokTile);
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s of wall time per wait
// Warps 0-3 hold the 128 TMEM lanes in the epilogue; warps 4..NI only issue
// MMAs.
static_assert(gemm_threads(kGemmIssuers / 2) >= 128, "the epilogue needs four warps");

struct GemmArgs {
  uint16_t *y;       // [m, n] BF16 bits
  int m, n;
  int h;             // weight rows per CTA (tile height), 1..kMmaM
  int kb_per_split;  // kBlockK-wide K blocks per CTA
  int stages;
  int bps;           // boxes per stage
  int splits;
  int l2_ahead;      // weight stages started towards L2 before the dependency wait
  // The GEMM enqueued after this one (tensor map tmap_pf): once this CTA's
  // last weight stage has landed, it starts towards L2 the first pf_stages
  // stages of the next GEMM's CTAs c, c + ctas, ... (c = this CTA's linear
  // index). pf_stages = 0: nothing.
  int pf_stages;
  int pf_h, pf_nkb, pf_bps, pf_tiles, pf_ctas;
  int x_ready;  // no running kernel writes x: copy it without waiting (the stores of y still wait)
};

// Bounded wait that also gives up as soon as another role raised `abort`.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile uint32_t *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Writes tile rows [r0, r1) of y (output features n0 + r0 ...; r1 - r0 and r0 a
// multiple of 8): the thread whose `row` is in [r0, r1) holds that row's 16
// token values in v (row < 0: none). The values are staged as BF16 in shared
// memory, then each token's row segment leaves in 16-byte stores (one per 8
// features) instead of one 2-byte store per token and feature. Called by all
// threads of the CTA.
template <int NT>
__device__ __forceinline__ void store_tile_rows(uint16_t *stage, const float (&v)[kTokTile], int r0,
                                                int r1, uint16_t *y, int n, int n0, int m, bool ok,
                                                int row) {
  const int tid = threadIdx.x, nr = r1 - r0;
  if (row >= r0 && row < r1) {
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) stage[t * nr + (row - r0)] = bf16_store_bits(v[t]);
  }
  __syncthreads();
  const int per_t = nr >> 3;
  for (int c = tid; c < m * per_t; c += NT) {
    const int t = c / per_t, q = c - t * per_t;
    const int row = n0 + r0 + 8 * q;
    if (ok && row < n)
      *reinterpret_cast<uint4 *>(y + static_cast<size_t>(t) * n + row) =
          *reinterpret_cast<const uint4 *>(stage + t * nr + 8 * q);
  }
}

// The GEMM epilogue after the accumulators are read: the split-K exchange
// between the S ranks of the cluster (S > 1), the optional output scale, the
// BF16 rounding (-0 stored as +0) and the stores of the tile's rows
// [n0, n0 + h) of y (each of rows 0..h-1 is held in acc by the one thread
// whose `row` it is; row < 0: the thread holds none). `stage` is idle shared
// memory for the row staging, `red` the exchange buffer counted on `red_bar`.
// Called by all NT threads of the CTA.
//
// Split-K across the S ranks of the cluster: rank r owns tile rows
// [r * R, (r + 1) * R). Every rank sends its FP32 partials of the rows it does
// not own to their owner (st.async into the owner's exchange buffer,
// red[q][row - r * R][t] for source rank q, counted on the owner's exchange
// barrier); the owner adds q = 0, 1, ..., S-1 in that order, its own partial
// taken from registers. A CTA leaves only after its exchange barrier has
// counted every byte its peers send it, so no peer writes into shared memory
// that is gone; one cluster barrier (before the first push) is enough.
template <int NT, bool kScaled>
__device__ __forceinline__ void splitk_store(const float (&acc)[kTokTile], float out_scale,
                                             uint16_t *stage, float *red, uint32_t red_bar,
                                             volatile uint32_t *abort_flag, bool aborted, int S,
                                             int h, uint16_t *y, int n, int n0, int m, int row) {
  const int tid = threadIdx.x;
  if (S == 1) {
    float v[kTokTile];
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) v[t] = kScaled ? __fmul_rn(acc[t], out_scale) : acc[t];
    // Outputs may still be read or written by the previous kernel in the stream.
    griddep_wait();
    store_tile_rows<NT>(stage, v, 0, h, y, n, n0, m, !aborted, row);
    return;
  }
  const int R = (h + S - 1) / S;
  const uint32_t rank = cluster_ctarank();
  const int lo = static_cast<int>(rank) * R;
  const int hi = min(h, lo + R);
  const int ng = (m + 3) / 4;  // groups of 4 tokens sent
  if (tid == 0)
    mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>((S - 1) * max(0, hi - lo) * ng * 16));
  cluster_wait();  // every peer's exchange barrier is initialised
  if (row >= 0 && row < h) {
    const uint32_t owner = static_cast<uint32_t>(row / R);
    if (owner != rank) {
      const int lr = row - static_cast<int>(owner) * R;
      const uint32_t dst =
          dsmem_map(smem_u32(red + (static_cast<int>(rank) * R + lr) * kTokTile), owner);
      const uint32_t rbar = dsmem_map(red_bar, owner);
#pragma unroll
      for (int g = 0; g < kTokTile / 4; ++g)
        if (g < ng)
          st_async_v4_f32(dst + 16 * g, acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3],
                          rbar);
    }
  }
  float v[kTokTile];
  if (row >= lo && row < hi) {
    if (!mbar_wait_bounded(red_bar, 0, kWaitLimitNs)) {
      atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
      *abort_flag = 1;
    }
    // All sums first, then the stores: a load issued after a global store
    // that the compiler cannot prove disjoint waits behind it.
    const int lr = row - lo;
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) v[t] = acc[t];
    if (rank != 0) {
      const float4 *r0 = reinterpret_cast<const float4 *>(red + lr * kTokTile);
#pragma unroll
      for (int g = 0; g < kTokTile / 4; ++g) {
        const float4 p = r0[g];
        v[4 * g] = p.x;
        v[4 * g + 1] = p.y;
        v[4 * g + 2] = p.z;
        v[4 * g + 3] = p.w;
      }
    }
    for (int q = 1; q < S; ++q) {
      if (q == static_cast<int>(rank)) {
#pragma unroll
        for (int t = 0; t < kTokTile; ++t) v[t] += acc[t];
      } else {
        const float4 *rq = reinterpret_cast<const float4 *>(red + (q * R + lr) * kTokTile);
#pragma unroll
        for (int g = 0; g < kTokTile / 4; ++g) {
          const float4 p = rq[g];
          v[4 * g] += p.x;
          v[4 * g + 1] += p.y;
          v[4 * g + 2] += p.z;
          v[4 * g + 3] += p.w;
        }
      }
    }
    if (kScaled) {
#pragma unroll
      for (int t = 0; t < kTokTile; ++t) v[t] = __fmul_rn(v[t], out_scale);
    }
  }
  __syncthreads();  // the exchange waits are over: *abort_flag is final
  const bool ok = !*abort_flag;
  // Outputs may still be read or written by the previous kernel in the
  // stream (the exchange above stays within this cluster's shared memory).
  griddep_wait();
  if ((R & 7) == 0) {
    store_tile_rows<NT>(stage, v, lo, hi > lo ? hi : lo, y, n, n0, m, ok, row);
  } else if (ok && row >= lo && row < hi && n0 + row < n) {
#pragma unroll
    for (int t = 0; t < kTokTile; ++t)
      if (t < m) y[static_cast<size_t>(t) * n + n0 + row] = bf16_store_bits(v[t]);
  }
}

// One CTA = h weight rows x one K slice of kb_per_split * 64 elements, moved
// args.bps 64-column boxes per pipeline stage.
// Warp 0 lane 0: TMA producer. Lane 0 of warps 1..NI: MMA issuers.
// Warp 2 owns the TMEM allocation. Warps 0-3 run the epilogue (one TMEM lane
// per thread; with the 64-row instruction, lanes 0-15 of each warp).
template <int NI>
__global__ void __launch_bounds__(gemm_threads(NI), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_pf, GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int B = args.bps;
  const int stages = args.stages;
  const int S = args.splits;
  const GemmLayout lay = gemm_layout(args.h, stages, B, S);
  const int slot_w = lay.slot_w;
  uint8_t *s_w = smem;                                     // stages*B weight slots
  uint8_t *s_x = smem + lay.x_off;                         // stages*B activation slots
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 2);
  float *red = reinterpret_cast<float *>(smem + lay.red_off);  // split-K exchange buffer
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = args.h;
  const int n0 = blockIdx.x * h;
  // Tiles of at most 64 rows: 64-row instructions, accumulator row r in TMEM
  // lane 32 * (r / 16) + r % 16; otherwise row r in lane r.
  const bool m64 = NI == kGemmIssuers && h <= 64;  // the launch pairs NI = 8 with h <= 64
  const uint32_t idesc = idesc_bf16_f32(m64 ? 64 : kMmaM, kTokTile);
  // Issuing warps: four reach the SM's floor for the 128-row instruction,
  // the 64-row one needs eight (the launch picks NI by the tile height).
  constexpr int ni = NI;
  constexpr uint32_t kCols = NI * kTokTile;  // TMEM columns, a power of two >= 32
  const int row = tid >= 128 ? -1 : !m64 ? tid : lane < 16 ? 16 * warp + lane : -1;
  const int nkb = args.kb_per_split;
  const int kb0 = blockIdx.y * nkb;
  const int nst = (nkb + B - 1) / B;                     // pipeline stages of work
  const uint32_t stage_tx = static_cast<uint32_t>(B * (h * 128 + kSlotXBytes));

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + stages);
  const uint32_t done_bar = smem_u32(bars + 2 * stages);
  const uint32_t red_bar = smem_u32(bars + 2 * stages + 1);  // peers' partials arrived

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, ni);  // one commit per issuer
    }
    mbar_init(done_bar, ni);
    mbar_init(red_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmap_w);
    tma_prefetch_map(&tmap_x);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // First phase of the cluster barrier: this CTA's exchange barrier is
  // initialised. Peers wait on it only before their first push, long after.
  if (S > 1) cluster_arrive();

  // Dependents may be scheduled as soon as every CTA of this grid is resident;
  // they order themselves after this grid with their own griddepcontrol.wait.
  griddep_launch_dependents();

  int issued = 0;
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------- TMA producer
    const uint64_t pol_w = l2_policy_evict_first();  // the weight is streamed once
    const uint64_t pol_x = l2_policy_evict_last();   // x is re-read by every row tile
    const int npre = nst < stages ? nst : stages;
    // One copy per operand and stage: the weight box is B blocks of h rows, the
    // activation box B blocks of 16 token rows (rows past m and blocks past K
    // arrive as zeros and count toward the transaction bytes all the same).
    // The weight is never written by another kernel: fill the ring with it
    // before waiting for the previous kernel in the stream.
    for (int i = 0; i < npre; ++i) {
      mbar_arrive_expect_tx(full0 + 8 * i, stage_tx);
      tma_load_3d(smem_u32(s_w + i * B * slot_w), &tmap_w, full0 + 8 * i, 0, n0, kb0 + i * B,
                  pol_w);
    }
    // and the next stages towards L2, while the previous kernel finishes
    for (int i = npre; i < nst && i < npre + args.l2_ahead; ++i)
      tma_prefetch_l2_3d(&tmap_w, 0, n0, kb0 + i * B);
    if (!args.x_ready) griddep_wait();
    for (int i = 0; i < npre; ++i)
      tma_load_3d(smem_u32(s_x + i * B * kSlotXBytes), &tmap_x, full0 + 8 * i, 0, 0, kb0 + i * B,
                  pol_x);
    issued = npre;
    for (int i = npre; i < nst; ++i) {
      const int s = i % stages;
      const uint32_t par = ((i / stages) & 1) ^ 1;
      if (!wait_or_abort(empty0 + 8 * s, par, abort_flag)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_PRODUCER);
        *abort_flag = 1;
        break;
      }
      const int kb = kb0 + i * B;
      mbar_arrive_expect_tx(full0 + 8 * s, stage_tx);
      tma_load_3d(smem_u32(s_w + s * B * slot_w), &tmap_w, full0 + 8 * s, 0, n0, kb, pol_w);
      tma_load_3d(smem_u32(s_x + s * B * kSlotXBytes), &tmap_x, full0 + 8 * s, 0, 0, kb, pol_x);
      issued = i + 1;
    }
    // Once this CTA's last stage has landed, HBM would idle here through the
    // epilogue, whatever runs in between and the next launch: start the next
    // GEMM's first weight stages towards L2. (Issued any earlier, these copies
    // delay the last stages of this GEMM, which every later kernel waits for.)
    if (args.pf_stages > 0 && !*abort_flag && issued > 0 &&
        mbar_wait_bounded(full0 + 8 * ((issued - 1) % stages), ((issued - 1) / stages) & 1,
                          kWaitLimitNs)) {
      const int ctas = static_cast<int>(gridDim.x * gridDim.y);
      for (int c = static_cast<int>(blockIdx.x + blockIdx.y * gridDim.x); c < args.pf_ctas; c += ctas) {
        const int pn0 = (c % args.pf_tiles) * args.pf_h;
        const int pkb0 = (c / args.pf_tiles) * args.pf_nkb;
        for (int j = 0; j < args.pf_stages && j * args.pf_bps < args.pf_nkb; ++j)
          tma_prefetch_l2_3d(&tmap_pf, 0, pn0, pkb0 + j * args.pf_bps);
      }
    }
  } else if (warp >= 1 && warp <= ni && lane == 0) {
    // ---------------------------------------------------- MMA issuers
    const int q = warp - 1;
    bool started = false;  // this issuer's accumulators hold a partial sum
    for (int i = 0; i < nst; ++i) {
      const int s = i % stages;
      const uint32_t par = (i / stages) & 1;
      if (!wait_or_abort(full0 + 8 * s, par, abort_flag)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_MMA);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      const int nb = min(B, nkb - i * B);
      for (int j = q; j < nb; j += ni) {
        const uint64_t adesc = smem_desc_k128(smem_u32(s_w + (s * B + j) * slot_w));
        const uint64_t bdesc = smem_desc_k128(smem_u32(s_x + (s * B + j) * kSlotXBytes));
#pragma unroll
        for (int kk = 0; kk < kBlockK / 16; ++kk) {
          // K advances 16 elements = 32 bytes inside the 128-byte swizzle row.
          tc_mma_bf16(tmem + static_cast<uint32_t>(acc_index(q, kk) * kTokTile), adesc + 2 * kk,
                      bdesc + 2 * kk, idesc, started || kk > 0);
        }
        started = true;
      }
      tc_commit(empty0 + 8 * s);  // this issuer's share of the stage has been read
    }
    tc_commit(done_bar);  // accumulators complete (or, after an abort, quiescent)
  }
  __syncwarp();

  // ------------------------------------------------------------ epilogue
  if (!mbar_wait_idle(done_bar, 0, kWaitLimitNs)) {
    atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
    *abort_flag = 1;
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    // Do not leave copies in flight into shared memory this CTA releases.
    const int first = issued > stages ? issued - stages : 0;
    for (int j = first; j < issued; ++j)
      mbar_wait_bounded(full0 + 8 * (j % stages), (j / stages) & 1, kWaitLimitNs);
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  tc_fence_after_sync();

  // After an abort the accumulators may still be written by MMAs in flight:
  // they are not read, and nothing is stored.
  float acc[kTokTile];
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) acc[t] = 0.0f;
  if (warp < 4 && !aborted)
    tmem_sum_accumulators<NI>(tmem + (static_cast<uint32_t>(warp * 32) << 16),
                                   acc_used(nkb, B, ni), acc);

  splitk_store<gemm_threads(NI), false>(acc, 1.0f, reinterpret_cast<uint16_t *>(s_w), red, red_bar,
                                    abort_flag, aborted, S, h, args.y, args.n, n0, args.m, row);

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    // The MMAs' final commit may not have arrived if the first wait ran out:
    // wait for it once more (bounded) before the columns are released.
    if (aborted && lane == 0 && !mbar_wait_idle(done_bar, 0, kWaitLimitNs))
      atomicOr(&g_device_status, SK_DEVICE_WAIT_TEARDOWN);
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kCols);
  }
}

// ----------------------------------------------------------------------------
// Weight-only NVFP4 GEMM: y[m, n] = bf16(w_scale * sum_k x[m, k] * W[n, k])
// with W held as e2m1 codes (two per byte, column 2c in the low nibble) and one
// e4m3 scale per 16 columns of a row, the NVFP4 layout of the pooler page's
// module docstring (cutedsl/moe/pooler_gather) applied to a weight. Not on the
// pages: it streams 4.5 bits per weight instead of 16.
//
// Roles (kW4Threads threads): warp 0 lane 0 issues the copies (codes and
// scales before the dependency wait, activations after it); lane 0 of warps
// 1..kW4Issuers issue the MMAs (K-step t of a block goes to issuer t mod 4,
// each with its own accumulator); warps kW4DeqWarp0.. expand the codes into a
// BF16 operand in tensor memory and put each block's activations in the
// order of that operand, in two groups that take alternate blocks (one
// group's barrier waits overlap the other's arithmetic); warps 0-3 run the
// epilogue. At 4.5 bits per weight the expansion (about three instructions
// per weight), not HBM and not the MMAs (an SM sustains one 128 x 16 x 16
// instruction per ~18 ns with A in tensor memory), bounds this kernel.
//
// Expansion. Placing an e2m1 code's three magnitude bits at bits 6..8 of a
// BF16 word and its sign at bit 15 gives the code's value times 2^-126
// (a subnormal for codes 1 and 9, whose exponent field is 0). One BF16 multiply
// by the block scale times 2^119 (exact in BF16 for every e4m3 value) then
// gives code * scale * 2^-7 exactly: at most six significant bits, within
// [2^-17, 21]. The epilogue multiplies the FP32 sum by w_scale * 2^7.
// Codes j and j + 4 of a 32-bit word (8 consecutive columns) sit 16 bits
// apart, so one shift-and-mask yields the BF16 pair (W[j], W[j + 4]); the
// operand therefore holds each group of 8 columns in the order
// 0, 4, 1, 5, 2, 6, 3, 7, and the activations are permuted the same way in
// shared memory (the dot product does not depend on the order of K).
constexpr int kW4Issuers = 4;
constexpr int kW4DeqWarp0 = 8;
constexpr int kW4DeqWarps = 16;
// The expansion warps form kW4DeqGroups groups that take alternate blocks, so
// that one group's barrier waits overlap another group's arithmetic. Within a
// group the warps of a TMEM lane quadrant split the block's 16 K-steps.
constexpr int kW4DeqGroups = 2;
constexpr int kW4GroupWarps = kW4DeqWarps / kW4DeqGroups;
constexpr int kW4StepsPerWarp = (kW4BlockK / 16) / (kW4GroupWarps / 4);
static_assert(kW4StepsPerWarp % 4 == 0, "a warp stores whole groups of 4 K-steps");
constexpr int kW4Threads = 32 * (kW4DeqWarp0 + kW4DeqWarps);
static_assert(kW4Issuers < kW4DeqWarp0, "issuer warps 1..kW4Issuers precede the expansion warps");
constexpr int kW4TmemCols = 512;  // accumulators at 0, A buffers at 128, 256, 384
static_assert(kW4ACols * (kW4ABufs + 1) <= kW4TmemCols, "tensor memory");
static_assert(kW4Issuers * kTokTile <= kW4ACols, "accumulators overlap the A buffers");
static_assert(kW4XBytes % (16 * kW4GroupWarps * 32) == 0, "activation chunks per expansion thread");

struct W4Args {
  uint16_t *y;             // [m, n] BF16 bits
  const float *w_scale;    // device FP32 [1]
  int m, n;
  int nblk;                // kW4BlockK-wide blocks per CTA (K slice)
  int stages, splits, l2_ahead;
};

// Bounded wait that also gives up once another role raised `abort`, for the
// roles of this kernel that share their SM's issue slots with the expansion
// warps: between polls the thread is suspended until the phase completes (or
// the hint runs out) instead of issuing instructions.
__device__ __forceinline__ bool w4_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 200000u)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// BF16 pair (scale * 2^119, scale * 2^119) of an e4m3 block scale, exact.
// The byte's exponent and mantissa placed at bits 20..26 of an FP32 word give
// |scale| * 2^-120 (an FP32 subnormal for subnormal scales); two exact
// multiplies by 2^120 and 2^119 give |scale| * 2^119, whose low 16 bits are
// zero (at most four significant bits), so its high half is the BF16 value.
// The sign bit is copied into both halves.
__device__ __forceinline__ uint32_t w4_scale_pair(uint32_t sf) {
  const float mag = __uint_as_float((sf & 0x7Fu) * (1u << 20));
  const uint32_t v = __float_as_uint(__fmul_rn(__fmul_rn(mag, 0x1p120f), 0x1p119f));
  const uint32_t sign = (sf & 0x80u) * 0x01000100u;  // bit 7 -> bits 15 and 31
  return __byte_perm(v, 0, 0x3232) | sign;
}

// The four BF16 pairs (W[j], W[j + 4]), j = 0..3, of 8 codes (code j in bits
// 4j..4j+3) times the scale pair c2, each an exact code * scale * 2^-7. Codes
// j and j + 4 sit 16 bits apart. Masking one such pair of nibbles and
// multiplying by 2^6 + 2^12 (2^2 + 2^8 for the odd nibbles) makes two copies
// of each nibble in disjoint bit ranges, one shifted so that its magnitude
// bits land at 6..8 and one so that its sign lands at 15; a second mask keeps
// just those. Codes 2, 3, 6, 7 go the same way after one right shift of the
// word.
__device__ __forceinline__ void w4_expand8(uint32_t w, uint32_t c2, uint32_t *o) {
  const uint32_t h = w >> 8;
  o[0] = mul_bf16x2(((w & 0x000F000Fu) * 4160u) & 0x81C081C0u, c2);
  o[1] = mul_bf16x2(((w & 0x00F000F0u) * 260u) & 0x81C081C0u, c2);
  o[2] = mul_bf16x2(((h & 0x000F000Fu) * 4160u) & 0x81C081C0u, c2);
  o[3] = mul_bf16x2(((h & 0x00F000F0u) * 260u) & 0x81C081C0u, c2);
}

__global__ void __launch_bounds__(kW4Threads, 1)
    gemm_nvfp4w_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_sf,
                       const __grid_constant__ CUtensorMap tmap_x, W4Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stages = args.stages;
  const int S = args.splits;
  const W4Layout lay = w4_layout(stages, S);
  uint8_t *s_q = smem;
  uint8_t *s_x = smem + lay.x_off;
  uint8_t *s_sf = smem + lay.sf_off;
  float *red = reinterpret_cast<float *>(smem + lay.red_off);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 2 * kW4ABufs + 2);
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kW4Rows;
  const int nblk = args.nblk;
  const int kb0 = blockIdx.y * nblk;
  const uint32_t stage_tx = static_cast<uint32_t>(kW4StageBytes);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + stages);
  const uint32_t afull0 = smem_u32(bars + 2 * stages);
  const uint32_t aempty0 = smem_u32(bars + 2 * stages + kW4ABufs);
  const uint32_t done_bar = smem_u32(bars + 2 * stages + 2 * kW4ABufs);
  const uint32_t red_bar = smem_u32(bars + 2 * stages + 2 * kW4ABufs + 1);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kW4Issuers);
    }
    for (int a = 0; a < kW4ABufs; ++a) {
      mbar_init(afull0 + 8 * a, kW4GroupWarps);
      mbar_init(aempty0 + 8 * a, kW4Issuers);
    }
    mbar_init(done_bar, kW4Issuers);
    mbar_init(red_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmap_q);
    tma_prefetch_map(&tmap_sf);
    tma_prefetch_map(&tmap_x);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), kW4TmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (S > 1) cluster_arrive();
  griddep_launch_dependents();

  int issued = 0;
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------- TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    const int npre = nblk < stages ? nblk : stages;
    for (int i = 0; i < npre; ++i) {
      mbar_arrive_expect_tx(full0 + 8 * i, stage_tx);
      tma_load_3d(smem_u32(s_q + i * kW4CodeBytes), &tmap_q, full0 + 8 * i, 0, n0, kb0 + i, pol_w);
      tma_load_3d(smem_u32(s_sf + i * kW4ScaleBytes), &tmap_sf, full0 + 8 * i, 0, n0, kb0 + i,
                  pol_w);
    }
    for (int i = npre; i < nblk && i < npre + args.l2_ahead; ++i) {
      tma_prefetch_l2_3d(&tmap_q, 0, n0, kb0 + i);
      tma_prefetch_l2_3d(&tmap_sf, 0, n0, kb0 + i);
    }
    griddep_wait();
    for (int i = 0; i < npre; ++i)
      tma_load_3d(smem_u32(s_x + i * kW4XBytes), &tmap_x, full0 + 8 * i, 0, 0, 4 * (kb0 + i),
                  pol_x);
    issued = npre;
    for (int i = npre; i < nblk; ++i) {
      const int s = i % stages;
      if (!w4_wait(empty0 + 8 * s, ((i / stages) & 1) ^ 1, abort_flag)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_PRODUCER);
        *abort_flag = 1;
        break;
      }
      const uint32_t fb = full0 + 8 * s;
      mbar_arrive_expect_tx(fb, stage_tx);
      tma_load_3d(smem_u32(s_q + s * kW4CodeBytes), &tmap_q, fb, 0, n0, kb0 + i, pol_w);
      tma_load_3d(smem_u32(s_sf + s * kW4ScaleBytes), &tmap_sf, fb, 0, n0, kb0 + i, pol_w);
      tma_load_3d(smem_u32(s_x + s * kW4XBytes), &tmap_x, fb, 0, 0, 4 * (kb0 + i), pol_x);
      issued = i + 1;
    }
  } else if (warp >= 1 && warp <= kW4Issuers && lane == 0) {
    // ---------------------------------------------------- MMA issuers
    const int q = warp - 1;
    bool started = false;
    for (int i = 0; i < nblk; ++i) {
      const int s = i % stages, a = i % kW4ABufs;
      if (!w4_wait(afull0 + 8 * a, (i / kW4ABufs) & 1, abort_flag)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_MMA);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t xs = smem_u32(s_x + s * kW4XBytes);
      const uint32_t acol = static_cast<uint32_t>(kW4ACols * (a + 1));
#pragma unroll
      for (int t = q; t < kW4BlockK / 16; t += kW4Issuers) {
        // K-step t: A columns acol + 8t; activations in 64-column box t / 4,
        // 32 bytes further per K-step inside the 128-byte swizzled row
        const uint64_t bdesc = smem_desc_k128(xs + (t / 4) * kSlotXBytes) + 2 * (t % 4);
        tc_mma_bf16_tmem_a(tmem + static_cast<uint32_t>(q * kTokTile), tmem + acol + 8 * t, bdesc,
                           kIdesc, started || t != q);
      }
      started = true;
      tc_commit(aempty0 + 8 * a);  // the A buffer has been read
      tc_commit(empty0 + 8 * s);   // and the stage's codes, scales and activations
    }
    tc_commit(done_bar);
  } else if (warp >= kW4DeqWarp0 && warp < kW4DeqWarp0 + kW4DeqWarps) {
    // ---------------------------------------------------- expansion (whole warps)
    const int dw = warp - kW4DeqWarp0;
    const int grp = dw / kW4GroupWarps;   // blocks grp, grp + kW4DeqGroups, ...
    const int gw = dw % kW4GroupWarps;    // warp within the group
    const int quad = warp & 3;            // TMEM lane quadrant this warp may access
    const int part = gw >> 2;             // K-steps part * kW4StepsPerWarp .. of each block
    const int row = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int kChunks = kW4StepsPerWarp / 2;  // 16-byte code chunks (2 K-steps each)
    constexpr int kXChunks = kW4XBytes / 16 / (kW4GroupWarps * 32);
    for (int i = grp; i < nblk; i += kW4DeqGroups) {
      const int s = i % stages, a = i % kW4ABufs;
      if (!w4_wait(full0 + 8 * s, (i / stages) & 1, abort_flag)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_MMA);
        *abort_flag = 1;
        break;
      }
      if (i >= kW4ABufs &&
          !w4_wait(aempty0 + 8 * a, ((i / kW4ABufs) - 1) & 1, abort_flag)) {
        atomicOr(&g_device_status, SK_DEVICE_WAIT_MMA);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      // Loads first: this row's codes of this warp's K-steps (16-byte chunks
      // of its 128-byte swizzled row), their scales, and this thread's share
      // of the block's activations.
      const uint32_t qrow = smem_u32(s_q + s * kW4CodeBytes) + row * 128;
      uint4 w[kChunks];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        w[c] = lds128(qrow + 16 * ((kChunks * part + c) ^ (row & 7)));
      uint32_t scw[kW4StepsPerWarp / 4];
#pragma unroll
      for (int j = 0; j < kW4StepsPerWarp / 4; ++j)
        scw[j] = lds32(smem_u32(s_sf + s * kW4ScaleBytes) + row * 16 + kW4StepsPerWarp * part + 4 * j);
      const uint32_t xs = smem_u32(s_x + s * kW4XBytes);
      uint4 xv[kXChunks];
#pragma unroll
      for (int j = 0; j < kXChunks; ++j)
        xv[j] = lds128(xs + 16 * (gw * 32 + lane + j * kW4GroupWarps * 32));
      // the block's activations in operand order: each 16-byte chunk of 8
      // columns x0..x7 becomes x0 x4 x1 x5 x2 x6 x3 x7 (chunks move whole
      // under the 128-byte swizzle)
#pragma unroll
      for (int j = 0; j < kXChunks; ++j) {
        uint4 o;
        o.x = __byte_perm(xv[j].x, xv[j].z, 0x5410);
        o.y = __byte_perm(xv[j].x, xv[j].z, 0x7632);
        o.z = __byte_perm(xv[j].y, xv[j].w, 0x5410);
        o.w = __byte_perm(xv[j].y, xv[j].w, 0x7632);
        sts128(xs + 16 * (gw * 32 + lane + j * kW4GroupWarps * 32), o);
      }
#pragma unroll
      for (int g = 0; g < kW4StepsPerWarp / 4; ++g) {  // groups of 4 K-steps
        uint32_t o[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {              // one 16-byte chunk = 2 K-steps
          const uint4 wc = w[2 * g + cc];
          const uint32_t c0 = w4_scale_pair((scw[g] >> (16 * cc)) & 0xFFu);
          const uint32_t c1 = w4_scale_pair((scw[g] >> (16 * cc + 8)) & 0xFFu);
          w4_expand8(wc.x, c0, o + 16 * cc);
          w4_expand8(wc.y, c0, o + 16 * cc + 4);
          w4_expand8(wc.z, c1, o + 16 * cc + 8);
          w4_expand8(wc.w, c1, o + 16 * cc + 12);
        }
        tmem_st_32x32b_x32(tmem + lane_base + kW4ACols * (a + 1) +
                               8 * (kW4StepsPerWarp * part + 4 * g),
                           o);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // the permuted activations, for the MMAs
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull0 + 8 * a);
    }
  }
  __syncwarp();

  // ------------------------------------------------------------ epilogue
  if (!mbar_wait_idle(done_bar, 0, kWaitLimitNs)) {
    atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
    *abort_flag = 1;
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    const int first = issued > stages ? issued - stages : 0;
    for (int j = first; j < issued; ++j)
      mbar_wait_bounded(full0 + 8 * (j % stages), (j / stages) & 1, kWaitLimitNs);
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  tc_fence_after_sync();

  float acc[kTokTile];
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) acc[t] = 0.0f;
  if (warp < 4 && !aborted)
    tmem_sum_accumulators<kW4Issuers>(tmem + (static_cast<uint32_t>(warp * 32) << 16), kW4Issuers,
                                      acc);
  // w_scale may have been written by the kernel ahead in the stream
  griddep_wait();
  const float out_scale = __fmul_rn(*args.w_scale, 128.0f);
  splitk_store<kW4Threads, true>(acc, out_scale, reinterpret_cast<uint16_t *>(s_q), red, red_bar,
                                 abort_flag, aborted, S, kW4Rows, args.y, args.n, n0, args.m,
                                 tid < kW4Rows ? tid : -1);

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    if (aborted && lane == 0 && !mbar_wait_idle(done_bar, 0, kWaitLimitNs))
      atomicOr(&g_device_status, SK_DEVICE_WAIT_TEARDOWN);
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kW4TmemCols);
  }
}

// ----------------------------------------------------------------------------
// Row reductions of the norm kernels. A token row is spread over a cluster of
// C CTAs (column chunks, one CTA per rank); each row sum is taken in a fixed
// order: each thread's own columns in column order, a shuffle-down tree inside
// each warp, the warp totals in warp order, then the CTA totals in rank order
// 0..C-1. Every rank pushes its CTA total into slot `rank` of every peer's
// shared memory with st.async (completing 4 bytes on the peer's mbarrier of
// that reduction), so each CTA ends with the same C values and forms the same
// sum. The order depends only on the row width and the launch shape, so the
// results are bitwise reproducible.
constexpr int kNormMaxCluster = 8;
constexpr int kNormReductions = 2;  // the dual norm takes two row sums

struct NormShared {
  uint64_t bar[kNormReductions];               // one mbarrier per row sum
  float part[kNormReductions][kNormMaxCluster];  // CTA totals by rank
  float red[32];                               // warp totals
  uint32_t abort;                              // a bounded wait ran out
};

// Initialises the exchange barriers (thread 0) and starts the cluster barrier
// that tells peers they may push (completed by norm_cluster_sum's first call).
__device__ __forceinline__ void norm_exchange_init(NormShared &sh, int C, int nred) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nred; ++i) {
      mbar_init(smem_u32(&sh.bar[i]), 1);
      // this CTA's single arrival, plus the bytes its C - 1 peers push
      mbar_arrive_expect_tx(smem_u32(&sh.bar[i]), static_cast<uint32_t>(4 * (C - 1)));
    }
    sh.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (C > 1) cluster_arrive();
}

// Sum of v over the CTA (every thread's v), then over the cluster's ranks in
// rank order; returned to every thread. `i` selects the reduction (its barrier
// and slots); the first call also completes the cluster barrier started by
// norm_exchange_init (peers' barriers are initialised before any push).
__device__ __forceinline__ float norm_cluster_sum(NormShared &sh, float v, int C, int i, bool first) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  if (nw > 1) {
    if (lane == 0) sh.red[warp] = v;
    __syncthreads();
    if (warp == 0) {
      v = lane < nw ? sh.red[lane] : 0.0f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
    }
  }
  const uint32_t rank = C > 1 ? cluster_ctarank() : 0;
  if (C > 1 && first) cluster_wait();
  if (threadIdx.x == 0) {
    sh.part[i][rank] = v;
    for (int q = 0; q < C; ++q) {
      if (q == static_cast<int>(rank)) continue;
      st_async_f32(dsmem_map(smem_u32(&sh.part[i][rank]), static_cast<uint32_t>(q)), v,
                   dsmem_map(smem_u32(&sh.bar[i]), static_cast<uint32_t>(q)));
    }
  }
  __syncthreads();  // this CTA's own slot is written; warp totals may be reused
  if (C > 1 && !mbar_wait_bounded(smem_u32(&sh.bar[i]), 0, kWaitLimitNs)) {
    atomicOr(&g_device_status, SK_DEVICE_WAIT_EPILOGUE);
    sh.abort = 1;
  }
  float t = 0.0f;
  for (int q = 0; q < C; ++q) t += sh.part[i][q];
  return t;
}

__device__ __forceinline__ float rms_inv(float sum, float n, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, n), eps)));
}

__device__ __forceinline__ void unpack8(const uint4 &v, uint16_t (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
    o[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
  }
}

__device__ __forceinline__ uint4 pack8(const uint16_t (&o)[8]) {
  uint4 v;
  v.x = o[0] | (static_cast<uint32_t>(o[1]) << 16);
  v.y = o[2] | (static_cast<uint32_t>(o[3]) << 16);
  v.z = o[4] | (static_cast<uint32_t>(o[5]) << 16);
  v.w = o[6] | (static_cast<uint32_t>(o[7]) << 16);
  return v;
}

// NVFP4 of one 16-element block of BF16 values (cutedsl/moe/pooler_gather:
// module docstring and nvfp4_compute_output_scale; the block-scale formula is
// our reading, (amax / 6) * gs, since the pages print only its inverse).
// Writes the 8 packed code bytes (column 2c in the low nibble) and returns the
// e4m3 scale byte. Every step is an IEEE FP32 operation.
__device__ __forceinline__ uint32_t nvfp4_block16(const uint16_t (&z)[16], float gs,
                                                  uint2 &packed) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(z[j])));
  const float t = __fmul_rn(__fdiv_rn(amax, 6.0f), gs);
  const uint32_t sf = cvt_f32_e4m3(t);
  const float sff = cvt_e4m3_f32(sf);
  const float os = (sff == 0.0f) ? 0.0f : __fdiv_rn(1.0f, __fmul_rn(sff, __fdiv_rn(1.0f, gs)));
  uint32_t b[8];
#pragma unroll
  for (int c = 0; c < 8; ++c)
    b[c] = cvt_f32x2_e2m1x2(__fmul_rn(bf16_bits_to_f32(z[2 * c]), os),
                            __fmul_rn(bf16_bits_to_f32(z[2 * c + 1]), os));
  packed.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  packed.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sf;
}

// Pre-expert RMSNorm + NVFP4 (cutedsl/moe/pooler_gather, module docstring;
// pooler_layer: weight applied after the norm). Grid (C, m), cluster (C, 1, 1):
// the C CTAs of a cluster share token row blockIdx.y, each thread owns one
// 16-column NVFP4 block (CTA r: blocks r * blockDim.x + threadIdx.x). With
// a == NULL the NVFP4 step is skipped and only z is stored: the norm of a BF16
// edge layer (same page, module docstring, ExpertsInputBf16).
__global__ void __launch_bounds__(1024)
    rmsnorm_nvfp4_kernel(const uint16_t *__restrict__ y, const uint16_t *__restrict__ norm_w,
                         float eps, float gc, const float *__restrict__ gs_ptr,
                         uint8_t *__restrict__ a, uint8_t *__restrict__ a_sf,
                         uint16_t *__restrict__ z_out, int n, int C) {
  __shared__ NormShared sh;
  const int row = blockIdx.y;
  const int blk = blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = blk < (n >> 4);
  griddep_launch_dependents();
  norm_exchange_init(sh, C, 1);

  uint16_t w[16];
  if (active) {  // the norm weight is never written by a kernel: read it before the wait
    const uint4 *wp = reinterpret_cast<const uint4 *>(norm_w + 16 * blk);
    uint16_t lo[8], hi[8];
    unpack8(__ldg(wp), lo);
    unpack8(__ldg(wp + 1), hi);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      w[j] = lo[j];
      w[8 + j] = hi[j];
    }
  }
  float gsv = 0.0f;
  griddep_wait();
  if (a && active) gsv = *gs_ptr;

  uint16_t v[16];
  float ss = 0.0f;
  if (active) {
    const uint4 *yp = reinterpret_cast<const uint4 *>(y + static_cast<size_t>(row) * n + 16 * blk);
    uint16_t lo[8], hi[8];
    unpack8(yp[0], lo);
    unpack8(yp[1], hi);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = lo[j];
      v[8 + j] = hi[j];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float f = bf16_bits_to_f32(v[j]);
      ss = __fmaf_rn(f, f, ss);
    }
  }
  const float r = rms_inv(norm_cluster_sum(sh, ss, C, 0, true), static_cast<float>(n), eps);

  if (active && !sh.abort) {
    uint16_t z[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float g = __fadd_rn(bf16_bits_to_f32(w[j]), gc);
      z[j] = bf16_store_bits(__fmul_rn(__fmul_rn(bf16_bits_to_f32(v[j]), r), g));
    }
    const size_t base = static_cast<size_t>(row) * n + 16 * blk;
    if (a) {  // NVFP4 layers; a BF16 edge layer stores z only
      uint2 packed;
      const uint32_t sf = nvfp4_block16(z, gsv, packed);
      reinterpret_cast<uint2 *>(a)[base >> 4] = packed;
      a_sf[base >> 4] = static_cast<uint8_t>(sf);
    }
    if (z_out) {
      uint16_t lo[8], hi[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        lo[j] = z[j];
        hi[j] = z[8 + j];
      }
      uint4 *zp = reinterpret_cast<uint4 *>(z_out + base);
      zp[0] = pack8(lo);
      zp[1] = pack8(hi);
    }
  }
}

// NVFP4 of a BF16 [m, n] tensor: one thread per 16-element block.
__global__ void __launch_bounds__(256)
    nvfp4_quantize_kernel(const uint16_t *__restrict__ z, const float *__restrict__ gs_ptr,
                          uint8_t *__restrict__ a, uint8_t *__restrict__ a_sf, int n) {
  griddep_launch_dependents();
  griddep_wait();
  const int row = blockIdx.y;
  const int blk = blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= (n >> 4)) return;
  const size_t base = static_cast<size_t>(row) * n + 16 * blk;
  const uint4 *zp = reinterpret_cast<const uint4 *>(z + base);
  uint16_t lo[8], hi[8], v[16];
  unpack8(zp[0], lo);
  unpack8(zp[1], hi);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = lo[j];
    v[8 + j] = hi[j];
  }
  uint2 packed;
  const uint32_t sf = nvfp4_block16(v, *gs_ptr, packed);
  reinterpret_cast<uint2 *>(a)[base >> 4] = packed;
  a_sf[base >> 4] = static_cast<uint8_t>(sf);
}

// Attention-boundary dual norm (cutedsl/oproj/batt, AttentionBoundary). Grid
// (C, m), cluster (C, 1, 1): the C CTAs of a cluster share token row
// blockIdx.y, each thread owns 8 consecutive columns (CTA r: chunks
// r * blockDim.x + threadIdx.x). The two row sums (of the partial, then of the
// updated residual) are cluster reductions. The elementwise steps use the
// packed FP32x2 operations (each lane an IEEE round-to-nearest operation, the
// same as the scalar one).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// the two BF16 of a 32-bit word as FP32 (low half first)
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

__global__ void __launch_bounds__(1024)
    dual_norm_kernel(const uint16_t *__restrict__ p, float *__restrict__ s,
                     const uint16_t *__restrict__ w1, float alpha,
                     const uint16_t *__restrict__ beta, const uint16_t *__restrict__ w2,
                     uint16_t *__restrict__ out, float eps_post, float eps_pre, float gc_post,
                     float gc_pre, int h, int C) {
  __shared__ NormShared sh;
  const int row = blockIdx.y;
  const int ch = blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = ch < (h >> 3);
  griddep_launch_dependents();
  norm_exchange_init(sh, C, 2);

  // Weights first (never written by a kernel), then wait for the producer of
  // the partial and of the residual stream.
  uint4 g1 = make_uint4(0, 0, 0, 0), gb = g1, g2 = g1;
  if (active) {
    if (w1) g1 = __ldg(reinterpret_cast<const uint4 *>(w1) + ch);
    gb = __ldg(reinterpret_cast<const uint4 *>(beta) + ch);
    g2 = __ldg(reinterpret_cast<const uint4 *>(w2) + ch);
  }
  griddep_wait();

  const size_t rbase = static_cast<size_t>(row) * h;
  float2 pv[4], sv[4];
  float ss1 = 0.0f;
  if (active) {
    const uint4 pw = reinterpret_cast<const uint4 *>(p + rbase)[ch];
    const float4 *sp = reinterpret_cast<const float4 *>(s + rbase) + 2 * ch;
    const float4 s0 = sp[0], s1 = sp[1];
    pv[0] = bf16x2_f2(pw.x);
    pv[1] = bf16x2_f2(pw.y);
    pv[2] = bf16x2_f2(pw.z);
    pv[3] = bf16x2_f2(pw.w);
    sv[0] = make_float2(s0.x, s0.y);
    sv[1] = make_float2(s0.z, s0.w);
    sv[2] = make_float2(s1.x, s1.y);
    sv[3] = make_float2(s1.z, s1.w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ss1 = __fmaf_rn(pv[j].x, pv[j].x, ss1);
      ss1 = __fmaf_rn(pv[j].y, pv[j].y, ss1);
    }
  }
  const float r1 = rms_inv(norm_cluster_sum(sh, ss1, C, 0, true), static_cast<float>(h), eps_post);

  float ss2 = 0.0f;
  if (active) {
    const uint32_t w1w[4] = {g1.x, g1.y, g1.z, g1.w};
    const uint32_t bw[4] = {gb.x, gb.y, gb.z, gb.w};
    const float2 r1v = make_float2(r1, r1), av = make_float2(alpha, alpha);
    const float2 gcv = make_float2(gc_post, gc_post);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 g = w1 ? __fadd2_rn(bf16x2_f2(w1w[j]), gcv) : make_float2(1.0f, 1.0f);
      const float2 q = __fmul2_rn(__fmul2_rn(pv[j], r1v), g);
      sv[j] = __ffma2_rn(bf16x2_f2(bw[j]), q, __fmul2_rn(av, sv[j]));
      ss2 = __fmaf_rn(sv[j].x, sv[j].x, ss2);
      ss2 = __fmaf_rn(sv[j].y, sv[j].y, ss2);
    }
    if (!sh.abort) {
      float4 *sp = reinterpret_cast<float4 *>(s + rbase) + 2 * ch;
      sp[0] = make_float4(sv[0].x, sv[0].y, sv[1].x, sv[1].y);
      sp[1] = make_float4(sv[2].x, sv[2].y, sv[3].x, sv[3].y);
    }
  }
  const float r2 = rms_inv(norm_cluster_sum(sh, ss2, C, 1, false), static_cast<float>(h), eps_pre);

  if (active && !sh.abort) {
    const uint32_t w2w[4] = {g2.x, g2.y, g2.z, g2.w};
    const float2 r2v = make_float2(r2, r2), gcv = make_float2(gc_pre, gc_pre);
    uint16_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = __fmul2_rn(__fmul2_rn(sv[j], r2v), __fadd2_rn(bf16x2_f2(w2w[j]), gcv));
      o[2 * j] = bf16_store_bits(v.x);
      o[2 * j + 1] = bf16_store_bits(v.y);
    }
    reinterpret_cast<uint4 *>(out + rbase)[ch] = pack8(o);
  }
}


// Waits on an mbarrier nothing completes, for at most limit_ns, with the
// bounded wait the kernels use; reports the expected timeout in the status word.
__global__ void wait_probe_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns)) atomicOr(&g_device_status, SK_DEVICE_WAIT_PROBE);
  }
}

// Format-conversion probe over n inputs (see sk_convert_probe).
__global__ void convert_probe_kernel(int kind, const void *__restrict__ in, void *__restrict__ out,
                                     int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (kind == 3) {
      static_cast<float *>(out)[i] = cvt_e4m3_f32(static_cast<const uint8_t *>(in)[i]);
      continue;
    }
    const float v = static_cast<const float *>(in)[i];
    if (kind == 0) {
      static_cast<uint8_t *>(out)[i] = static_cast<uint8_t>(cvt_f32x2_e2m1x2(v, 0.0f) & 0xFu);
    } else if (kind == 1) {
      static_cast<uint8_t *>(out)[i] = static_cast<uint8_t>(cvt_f32_e4m3(v));
    } else {
      static_cast<uint16_t *>(out)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
}

// ---------------------------------------------------------------- host side
size_t gemm_smem_bytes(int h, int stages, int bps, int splits) {
  return 1024 + static_cast<size_t>(gemm_layout(h, stages, bps, splits).total);
}

namespace {
std::mutex g_setup_mutex;
DeviceInfo g_info[64];
bool g_ready[64];

template <typename... Args>
cudaError_t launch_ex(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, bool pdl, dim3 cluster,
                      typename std::remove_reference<Args>::type... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = cluster.x;
    attrs[na].val.clusterDim.y = cluster.y;
    attrs[na].val.clusterDim.z = cluster.z;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
}  // namespace

cudaError_t device_setup(int device, DeviceInfo *info) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_ready[device]) {
    DeviceInfo d;
    cudaError_t e;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device))) return e;
    d.sm_count = v;
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, device))) return e;
    if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, device))) return e;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, device))) return e;
    d.max_smem_optin = static_cast<size_t>(v);
    if (d.major == 10 && d.minor == 3) {
      // dynamic shared memory up to the opt-in limit less each kernel's static part
      cudaFuncAttributes fa;
      for (auto *kern : {gemm_kernel<kGemmIssuers / 2>, gemm_kernel<kGemmIssuers>}) {
        if ((e = cudaFuncGetAttributes(&fa, kern))) return e;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(d.max_smem_optin - fa.sharedSizeBytes))))
          return e;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)))
          return e;
      }
      if ((e = cudaFuncGetAttributes(&fa, gemm_nvfp4w_kernel))) return e;
      if ((e = cudaFuncSetAttribute(gemm_nvfp4w_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(d.max_smem_optin - fa.sharedSizeBytes))))
        return e;
      if ((e = cudaFuncSetAttribute(gemm_nvfp4w_kernel,
                                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1)))
        return e;
    }
    g_info[device] = d;
    g_ready[device] = true;
  }
  *info = g_info[device];
  return cudaSuccess;
}

int gemm_max_clusters(int device, int splits, int ctas_per_sm, int h) {
  static std::mutex mu;
  static int cache[64][5][2][2];
  int idx = 0;
  while ((1 << idx) < splits && idx < 4) ++idx;
  const int per = ctas_per_sm >= 2 ? 1 : 0;
  const int ni = gemm_issuers(h);
  const int wide = ni == kGemmIssuers ? 1 : 0;
  if (device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[device][idx][per][wide] == 0) {
    int clusters = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, splits, 1);
    cfg.blockDim = dim3(gemm_threads(ni));
    // more than half an SM's shared memory: one CTA per SM; else two
    cfg.dynamicSmemBytes = per ? 100 * 1024 : 120 * 1024;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = static_cast<unsigned>(splits);
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t oe = wide ? cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel<kGemmIssuers>, &cfg)
                                : cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel<kGemmIssuers / 2>, &cfg);
    if (oe != cudaSuccess || clusters < 1) clusters = -1;
    cache[device][idx][per][wide] = clusters;
  }
  return cache[device][idx][per][wide];
}

cudaError_t launch_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, uint16_t *y, int m,
                        int n, int k, int splits, int h, int stages, int bps,
                        cudaStream_t stream, bool pdl, const GemmPrefetch *pf, int l2_ahead,
                        bool x_ready) {
  if (h % 8 || h < 8 || h > kMmaM || bps < 1 || bps > kMaxBoxesPerStage) return cudaErrorInvalidValue;
  GemmArgs a = {};
  a.y = y;
  a.m = m;
  a.n = n;
  a.h = h;
  a.kb_per_split = k / (kBlockK * splits);
  a.stages = stages;
  a.bps = bps;
  a.splits = splits;
  // Weight stages started towards L2 before the dependency wait, beyond the
  // ring: by default about 256 KiB per CTA (measured best for GEMMs that
  // follow one another: the previous kernel's tail leaves HBM idle; much
  // more slows the memory accesses of a norm kernel between two GEMMs), or
  // what the caller says (l2_ahead >= 0). SK_L2_AHEAD overrides both.
  {
    const char *v = std::getenv("SK_L2_AHEAD");
    const int stage_w = bps * h * 128;
    a.l2_ahead = v ? std::atoi(v) : l2_ahead >= 0 ? l2_ahead : (256 * 1024 + stage_w - 1) / stage_w;
    if (a.l2_ahead < 0) a.l2_ahead = 0;
    if (a.l2_ahead > 64) a.l2_ahead = 64;
  }
  a.x_ready = x_ready ? 1 : 0;
  if (pf && pf->stages > 0) {
    if (pf->h % 8 || pf->h < 8 || pf->h > kMmaM || pf->bps < 1 || pf->bps > kMaxBoxesPerStage ||
        pf->tiles < 1 || pf->splits < 1 || pf->nkb < 1)
      return cudaErrorInvalidValue;
    a.pf_stages = pf->stages;
    a.pf_h = pf->h;
    a.pf_nkb = pf->nkb;
    a.pf_bps = pf->bps;
    a.pf_tiles = pf->tiles;
    a.pf_ctas = pf->tiles * pf->splits;
  }
  const dim3 grid((n + h - 1) / h, splits, 1);
  const size_t smem = gemm_smem_bytes(h, stages, bps, splits);
  const CUtensorMap &tmap_pf = a.pf_stages ? pf->map : tmap_w;
  if (gemm_issuers(h) == kGemmIssuers)
    return launch_ex(gemm_kernel<kGemmIssuers>, grid, dim3(gemm_threads(kGemmIssuers)), smem, stream,
                     pdl, dim3(1, splits, 1), tmap_w, tmap_x, tmap_pf, a);
  return launch_ex(gemm_kernel<kGemmIssuers / 2>, grid, dim3(gemm_threads(kGemmIssuers / 2)), smem,
                   stream, pdl, dim3(1, splits, 1), tmap_w, tmap_x, tmap_pf, a);
}

// Cluster size and CTA width of a norm over `units` per row (NVFP4 blocks or
// 8-column chunks): up to kNormMaxCluster CTAs per row, each with at least
// `min_per_cta` units, whole warps.
static void norm_shape(int units, int min_per_cta, int *C, int *threads) {
  int c = (units + min_per_cta - 1) / min_per_cta;
  c = c < 1 ? 1 : (c > kNormMaxCluster ? kNormMaxCluster : c);
  const int per = (units + c - 1) / c;
  *C = c;
  *threads = (per + 31) / 32 * 32;
}

size_t w4_smem_bytes(int stages, int splits) {
  const size_t b = 1024 + static_cast<size_t>(w4_layout(stages, splits).total);
  return b < kW4MinSmem ? kW4MinSmem : b;
}

int w4_max_clusters(int device, int splits) {
  static std::mutex mu;
  static int cache[64][5];
  int idx = 0;
  while ((1 << idx) < splits && idx < 4) ++idx;
  if (device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[device][idx] == 0) {
    int clusters = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, splits, 1);
    cfg.blockDim = dim3(kW4Threads);
    cfg.dynamicSmemBytes = w4_smem_bytes(kW4MaxStages, splits);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = static_cast<unsigned>(splits);
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_nvfp4w_kernel, &cfg) != cudaSuccess ||
        clusters < 1)
      clusters = -1;
    cache[device][idx] = clusters;
  }
  return cache[device][idx];
}

cudaError_t launch_gemm_nvfp4w(const CUtensorMap &tmap_q, const CUtensorMap &tmap_sf,
                               const CUtensorMap &tmap_x, const float *w_scale, uint16_t *y,
                               int m, int n, int k, int splits, int stages, int l2_ahead,
                               cudaStream_t stream, bool pdl) {
  if (stages < 1 || stages > kW4MaxStages || splits < 1 || k % (kW4BlockK * splits))
    return cudaErrorInvalidValue;
  W4Args a = {};
  a.y = y;
  a.w_scale = w_scale;
  a.m = m;
  a.n = n;
  a.nblk = k / (kW4BlockK * splits);
  a.stages = stages < a.nblk ? stages : a.nblk;
  // A ring slot reused within the slice must be consumed by one expansion
  // group only (blocks alternate between the groups), so that every wait on
  // its barrier is for the next phase: an even number of stages.
  if (a.stages < a.nblk && a.stages % kW4DeqGroups) a.stages -= a.stages % kW4DeqGroups;
  if (a.stages < kW4DeqGroups && a.nblk > a.stages) a.stages = kW4DeqGroups;
  a.splits = splits;
  a.l2_ahead = l2_ahead < 0 ? 0 : (l2_ahead > 64 ? 64 : l2_ahead);
  const dim3 grid((n + kW4Rows - 1) / kW4Rows, splits, 1);
  return launch_ex(gemm_nvfp4w_kernel, grid, dim3(kW4Threads), w4_smem_bytes(a.stages, splits),
                   stream, pdl, dim3(1, splits, 1), tmap_q, tmap_sf, tmap_x, a);
}

cudaError_t launch_rmsnorm_nvfp4(const uint16_t *y, const uint16_t *norm_w, float eps, float gc,
                                 const float *gs, uint8_t *a, uint8_t *a_sf, uint16_t *z_out,
                                 int m, int n, cudaStream_t stream, bool pdl) {
  // one thread per 16-column block, a cluster of CTAs per token row
  // (n <= 16384: at most 1024 blocks over at most 8 CTAs), at least 64 blocks
  // per CTA: at n = 4096, 4 CTAs of 64 threads (measured on GB300 against 8
  // of 32: the pooler call 13.8 against 14.6 us at b = 8, the decode chain
  // 0.03 us per layer faster; the wait for the cluster's slowest CTA is
  // shorter with fewer of them)
  int C, threads;
  norm_shape(n / 16, 64, &C, &threads);
  return launch_ex(rmsnorm_nvfp4_kernel, dim3(C, m), dim3(threads), 0, stream, pdl, dim3(C, 1, 1),
                   y, norm_w, eps, gc, gs, a, a_sf, z_out, n, C);
}

cudaError_t launch_nvfp4_quantize(const uint16_t *z, const float *gs, uint8_t *a, uint8_t *a_sf,
                                  int m, int n, cudaStream_t stream, bool pdl) {
  const int nblk = n / 16;
  const dim3 grid((nblk + 255) / 256, m);
  return launch_ex(nvfp4_quantize_kernel, grid, dim3(256), 0, stream, pdl, dim3(1, 1, 1), z, gs, a,
                   a_sf, n);
}

cudaError_t launch_dual_norm(const uint16_t *p, float *s, const uint16_t *w1, float alpha,
                             const uint16_t *beta, const uint16_t *w2, uint16_t *out,
                             float eps_post, float eps_pre, float gc_post, float gc_pre, int m,
                             int h, cudaStream_t stream, bool pdl) {
  // 8 columns per thread, a cluster of CTAs per token row (h <= 8192 is
  // checked by the caller: at most 1024 chunks over at most 8 CTAs)
  int C, threads;
  norm_shape(h / 8, 128, &C, &threads);
  return launch_ex(dual_norm_kernel, dim3(C, m), dim3(threads), 0, stream, pdl, dim3(C, 1, 1), p,
                   s, w1, alpha, beta, w2, out, eps_post, eps_pre, gc_post, gc_pre, h, C);
}

cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_convert_probe(int kind, const void *in, void *out, int n, cudaStream_t stream) {
  int blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  convert_probe_kernel<<<blocks, 256, 0, stream>>>(kind, in, out, n);
  return cudaGetLastError();
}

cudaError_t read_device_status(uint32_t *out, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e) return e;
  if ((e = cudaMemcpyFromSymbol(out, g_device_status, sizeof(uint32_t)))) return e;
  if (clear) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t)))) return e;
  }
  return cudaSuccess;
}

}  // namespace sk

