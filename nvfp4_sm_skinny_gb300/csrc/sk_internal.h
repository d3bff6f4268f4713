// Internal interface between the C-ABI front end (sk_api.cu) and the kernel
// translation unit (sk_kernels.cu). Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sk.h"

namespace sk {

// Records `msg` as this thread's sk_last_error() and returns `st`.
sk_status report_error(sk_status st, const char *msg);

// GEMM tiling. Each CTA owns h <= kMmaM consecutive weight rows (output
// features) and one K slice. The tensor-core instruction is M = kMmaM weight
// rows by N = kTokTile token columns by K = 16 (rows of x beyond m are
// zero-filled by the copy engine; tile rows beyond h hold stale data whose
// accumulator lanes are never stored). Each pipeline stage moves `bps` boxes
// of kBlockK columns (1 <= bps <= kMaxBoxesPerStage, chosen per launch): a
// weight box of h rows (its slot is h rounded up to 8 rows, 1 KiB per 8 rows)
// and an activation box of 16 rows. A stage is one mbarrier round trip between
// the copy engine and the MMA issuer; with one CTA per SM that round trip, not
// the bytes, bounds the stream unless stages are large, so the planner makes
// them as large as the ring allows while keeping at least three in flight.
constexpr int kMmaM = 128;
constexpr int kTokTile = 16;
constexpr int kBlockK = 64;
constexpr int kMaxBoxesPerStage = 8;
constexpr int kSlotXBytes = kTokTile * kBlockK * 2;  // 2 KiB
constexpr int kMmaABytes = kMmaM * kBlockK * 2;      // 16 KiB read by one MMA row block
constexpr int kMaxStages = 16;
// MMA issue. One thread issuing tcgen05.mma is held ~144 ns per instruction
// whatever its M (64, 128) and N (16 to 256); an SM's floor is set by the
// shared-memory reads of the operands (~105 B per clock: ~22 ns per
// 128 x 16 x 16 instruction, 4.5 KiB, reached from four issuing warps; ~12 ns
// per 64 x 16 x 16, 2.5 KiB, which takes about eight), measured on GB300. So
// a CTA issues from NI warps (four for 128-row tiles, kGemmIssuers = eight
// for tiles of at most 64 rows): box j of a stage goes to issuer j mod NI,
// and issuer q accumulates into its own TMEM accumulator (16 FP32
// columns), first written by the issuer's first box of the slice. The
// epilogue adds the used accumulators in index order, so the sum order is
// fixed. Tiles of at most 64 rows use the 64-row instruction (half the
// operand reads); its accumulator row r sits in TMEM lane 32 * (r / 16) +
// r % 16.
constexpr int kGemmIssuers = 8;                 // the most issuing warps of a launch
constexpr int kNumAcc = kGemmIssuers;           // one accumulator per issuer
// The kernel is built for NI = 4 (128-row tiles) and NI = 8 (tiles of at most
// 64 rows): 32 * (1 + NI) threads, NI * kTokTile TMEM columns.
__host__ __device__ constexpr int gemm_issuers(int h) { return h <= 64 ? kGemmIssuers : kGemmIssuers / 2; }
__host__ __device__ constexpr int gemm_threads(int ni) { return 32 * (1 + ni); }
__host__ __device__ constexpr int acc_index(int q, int /*kk*/) { return q; }
// Accumulators written by a K slice of nkb boxes moved bps per stage by ni
// issuers: those of the issuers that own a box of the first stage.
__host__ __device__ inline int acc_used(int nkb, int bps, int ni) {
  int b = nkb < bps ? nkb : bps;
  if (b > ni) b = ni;
  return b;
}
// Shared memory per CTA when two CTAs share an SM.
constexpr size_t kTwoPerSmSmem = 110 * 1024;
// Shared memory per CTA when one CTA owns an SM.
constexpr size_t kOnePerSmSmem = 226 * 1024;

// Shared-memory layout of a GEMM CTA, relative to its 1024-aligned base:
// weight slots [0, x_off), activation slots [x_off, red_off) (the data region
// also covers the 16 KiB an MMA reads from the last weight slot), the split-K
// exchange buffer [red_off, bar_off) that peers of the cluster write into
// while this CTA may still be streaming (S ranks x R rows x 16 tokens FP32,
// R = ceil(h / S)), then the mbarriers.
struct GemmLayout {
  int slot_w;  // bytes per weight slot
  int x_off;   // first activation slot
  int red_off; // split-K exchange buffer
  int bar_off; // mbarriers (2 * stages + 2), then the TMEM address and a flag
  int total;   // bytes from the aligned base to the end of the flag words
};

__host__ __device__ inline GemmLayout gemm_layout(int h, int stages, int bps, int splits) {
  GemmLayout L;
  L.slot_w = ((h + 7) / 8) * 1024;
  const int nslot = stages * bps;
  L.x_off = nslot * L.slot_w;
  int end = L.x_off + nslot * kSlotXBytes;
  const int mma_end = (nslot - 1) * L.slot_w + kMmaABytes;
  if (mma_end > end) end = mma_end;
  L.red_off = (end + 15) / 16 * 16;
  const int rows = splits > 1 ? splits * ((h + splits - 1) / splits) : 0;
  L.bar_off = L.red_off + rows * kTokTile * 4;
  L.total = L.bar_off + (2 * stages + 2) * 8 + 8;
  return L;
}

// Weight-only NVFP4 GEMM tiling. A CTA owns kW4Rows weight rows (the MMA's M)
// and one K slice, moved in blocks of kW4BlockK columns: per block the copy
// engine brings 128 code bytes and 16 scale bytes per row and the block's
// 16 x 256 BF16 activations; dequantization warps expand the codes into BF16
// tensor-memory operands (kW4ACols columns per block, kW4ABufs buffers).
constexpr int kW4BlockK = 256;
constexpr int kW4Rows = 128;
constexpr int kW4CodeBytes = kW4Rows * kW4BlockK / 2;   // 16 KiB
constexpr int kW4ScaleBytes = kW4Rows * kW4BlockK / 16; // 2 KiB
constexpr int kW4XBytes = kTokTile * kW4BlockK * 2;     // 8 KiB
constexpr int kW4StageBytes = kW4CodeBytes + kW4ScaleBytes + kW4XBytes;
constexpr int kW4ABufs = 3;
constexpr int kW4ACols = kW4BlockK / 2;                 // 128
constexpr int kW4MaxStages = 8;
// At least this much dynamic shared memory per CTA, so that two CTAs of the
// kernel never share an SM (each allocates all of the SM's tensor memory).
constexpr size_t kW4MinSmem = 116 * 1024;

// Shared-memory layout of a weight-only NVFP4 GEMM CTA, from its 1024-aligned
// base: code slots (16 KiB each, 128-byte swizzled rows), activation slots
// (8 KiB), scale slots (2 KiB), the split-K exchange buffer, the mbarriers.
struct W4Layout {
  int x_off, sf_off, red_off, bar_off, total;
};

__host__ __device__ inline W4Layout w4_layout(int stages, int splits) {
  W4Layout L;
  L.x_off = stages * kW4CodeBytes;
  L.sf_off = L.x_off + stages * kW4XBytes;
  L.red_off = L.sf_off + stages * kW4ScaleBytes;
  const int rows = splits > 1 ? splits * ((kW4Rows + splits - 1) / splits) : 0;
  L.bar_off = L.red_off + rows * kTokTile * 4;
  // full[stages], empty[stages], a_full[3], a_empty[3], done, exchange; then
  // the TMEM address and an abort flag
  L.total = L.bar_off + (2 * stages + 2 * kW4ABufs + 2) * 8 + 8;
  return L;
}

struct DeviceInfo {
  int sm_count = 0;
  int major = 0, minor = 0;
  size_t max_smem_optin = 0;
};

// Per-device properties and one-time kernel attribute set-up for the current
// device. Returns cudaSuccess or the first error.
cudaError_t device_setup(int device, DeviceInfo *info);

// Dynamic shared memory of a GEMM CTA with tile height h, `stages` stages of
// `bps` boxes and `splits` cluster ranks.
size_t gemm_smem_bytes(int h, int stages, int bps, int splits);

// Largest number of clusters of `splits` GEMM CTAs that can be resident at
// once with `ctas_per_sm` (1 or 2) GEMM CTAs per SM (cached).
int gemm_max_clusters(int device, int splits, int ctas_per_sm, int h = kMmaM);

// The GEMM enqueued next, whose first weight stages a GEMM launch starts
// towards L2 once it has issued its own last weight copy: its weight map (3-D,
// box {64, h, bps}), tile height, K blocks per split, boxes per stage, row
// tiles and splits, and how many of its stages to start per CTA.
struct GemmPrefetch {
  CUtensorMap map;
  int h, nkb, bps, tiles, splits, stages;
};

// Launches the split-K GEMM: grid (ceil(n / h), splits), cluster
// (1, splits, 1); tile height h rows, `stages` pipeline stages of `bps` boxes.
// pf (may be null): the next GEMM's weights to start towards L2. l2_ahead:
// own weight stages beyond the ring started towards L2 before the dependency
// wait (-1: about 256 KiB). x_ready: the previous kernel does not write x, so
// its copies do not wait for that kernel (the stores of y still do).
cudaError_t launch_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, uint16_t *y, int m,
                        int n, int k, int splits, int h, int stages, int bps, cudaStream_t stream,
                        bool pdl, const GemmPrefetch *pf = nullptr, int l2_ahead = -1,
                        bool x_ready = false);

// Dynamic shared memory of a weight-only NVFP4 GEMM CTA.
size_t w4_smem_bytes(int stages, int splits);

// Largest number of clusters of `splits` weight-only NVFP4 GEMM CTAs that can
// be resident at once (one CTA per SM; cached).
int w4_max_clusters(int device, int splits);

// Launches the weight-only NVFP4 GEMM: grid (ceil(n / 128), splits), cluster
// (1, splits, 1). tmap_q: codes {128 bytes, n rows, k / 256 blocks}, box
// {128, 128, 1}, 128-byte swizzle; tmap_sf: scales {16 bytes, n, k / 256},
// box {16, 128, 1}; tmap_x: activations {64, m, k / 64}, box {64, 16, 4}.
cudaError_t launch_gemm_nvfp4w(const CUtensorMap &tmap_q, const CUtensorMap &tmap_sf,
                               const CUtensorMap &tmap_x, const float *w_scale, uint16_t *y,
                               int m, int n, int k, int splits, int stages, int l2_ahead,
                               cudaStream_t stream, bool pdl);

cudaError_t launch_rmsnorm_nvfp4(const uint16_t *y, const uint16_t *norm_w, float eps, float gc,
                                 const float *gs, uint8_t *a, uint8_t *a_sf, uint16_t *z_out,
                                 int m, int n, cudaStream_t stream, bool pdl);

cudaError_t launch_nvfp4_quantize(const uint16_t *z, const float *gs, uint8_t *a, uint8_t *a_sf,
                                  int m, int n, cudaStream_t stream, bool pdl);

cudaError_t launch_dual_norm(const uint16_t *p, float *s, const uint16_t *w1, float alpha,
                             const uint16_t *beta, const uint16_t *w2, uint16_t *out,
                             float eps_post, float eps_pre, float gc_post, float gc_pre, int m,
                             int h, cudaStream_t stream, bool pdl);

cudaError_t launch_convert_probe(int kind, const void *in, void *out, int n, cudaStream_t stream);

cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t stream);

cudaError_t read_device_status(uint32_t *out, bool clear);

// The current device, checked to be compute capability 10.3, set up.
sk_status checked_device(DeviceInfo *info, int *device);
bool pdl_on();

}  // namespace sk
