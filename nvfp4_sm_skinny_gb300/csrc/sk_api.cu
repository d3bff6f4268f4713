// C-ABI front end of libsk: argument validation (before any CUDA call), the
// device check, TMA descriptor encoding, split-count choice and kernel chaining.
// Validation mirrors the unpooler page's Unpooler.unsupported, Unpooler.run and
// launch_unsupported: shape, dtype (here: the caller's contract), contiguity
// and 16-byte alignment are checked before launch and reported as a reason
// string.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "sk.h"
#include "sk_internal.h"

namespace {

thread_local std::string t_last_error;

sk_status fail(sk_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

sk_status ok() {
  t_last_error.clear();
  return SK_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pdl_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("SK_NO_PDL");
    return !(v && v[0] && v[0] != '0');
  }();
  return on;
}

// Current device, checked to be compute capability 10.3, with its one-time
// set-up done.
sk_status current_device(sk::DeviceInfo *info) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SK_ERR_CUDA, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (std::getenv("SK_FORCE_ARCH_FAIL"))
    return fail(SK_ERR_ARCH, "device %d rejected (SK_FORCE_ARCH_FAIL is set)", dev);
  e = sk::device_setup(dev, info);
  if (e != cudaSuccess)
    return fail(SK_ERR_CUDA, "device %d set-up failed: %s", dev, cudaGetErrorString(e));
  if (info->major != 10 || info->minor != 3)
    return fail(SK_ERR_ARCH, "libsk needs a compute capability 10.3 GPU (GB300); device %d is %d.%d",
                dev, info->major, info->minor);
  return SK_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a row-major BF16 matrix [rows, cols] seen as three
// dimensions {64 columns, rows, cols / 64 blocks}: one box is `box_blocks`
// consecutive 64-column blocks of `box_rows` rows, landing in shared memory as
// box_blocks tiles of box_rows x 128 bytes, each with the 128-byte swizzle the
// MMA descriptors expect (box_rows a multiple of 8 keeps every tile 1 KiB
// aligned). Rows past `rows` and blocks past cols / 64 read as zero.
sk_status make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows,
                   int box_blocks) {
  auto fn = encode_fn();
  if (!fn) return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(sk::kBlockK), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(cols / sk::kBlockK)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, sk::kBlockK * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(sk::kBlockK), static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(box_blocks)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return SK_OK;
}

// Tensor map of NVFP4 weight bytes [rows, row_bytes] seen as three dimensions
// {box_bytes, rows, row_bytes / box_bytes}: one box is box_bytes of each of
// `box_rows` rows of one K block, 128-byte swizzled when `swizzle` (the code
// tile whose rows the expansion warps read) or plain (the scale tile). Rows
// past `rows` read as zero.
sk_status make_byte_map(CUtensorMap *map, const void *base, int rows, int row_bytes, int box_bytes,
                        int box_rows, bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(box_bytes), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(row_bytes / box_bytes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(box_bytes)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_bytes), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return SK_OK;
}

sk_status check_gemm_shape(int m, int n, int k, int splits) {
  if (m < 1 || m > SK_MAX_M)
    return fail(SK_ERR_INVALID_ARG, "m=%d: needs 1 <= m <= %d token rows", m, SK_MAX_M);
  if (n <= 0 || n % 16)
    return fail(SK_ERR_INVALID_ARG, "n=%d: needs a positive multiple of 16 output features", n);
  if (k <= 0 || k % sk::kBlockK)
    return fail(SK_ERR_INVALID_ARG, "k=%d: needs a positive multiple of %d", k, sk::kBlockK);
  if (splits != 0 && splits != 1 && splits != 2 && splits != 4 && splits != 8 && splits != 16)
    return fail(SK_ERR_UNSUPPORTED, "unsupported split count %d (0, 1, 2, 4, 8 or 16)", splits);
  if (splits > 0 && k % (sk::kBlockK * splits))
    return fail(SK_ERR_UNSUPPORTED, "K=%d does not split into %d slices of whole %d-wide blocks", k,
                splits, sk::kBlockK);
  return SK_OK;
}

// Launch plan of the GEMM for one shape.
struct GemmPlan {
  int splits;  // K slices (cluster ranks)
  int h;       // weight rows per CTA
  int stages;  // pipeline stages per CTA
  int bps;     // 64-column boxes per stage
};

int env_int(const char *name, int lo, int hi) {
  const char *v = std::getenv(name);
  if (!v || !v[0]) return 0;
  const int x = std::atoi(v);
  return (x >= lo && x <= hi) ? x : 0;
}

// Ring shape for a K slice of nkb boxes: the largest boxes-per-stage count that
// still leaves three stages in flight (or holds the whole slice), then as many
// stages as the shared-memory budget holds. SK_BPS / SK_STAGES override.
template <typename Bytes>
void choose_ring(int nkb, size_t budget, Bytes bytes, int *stages, int *bps) {
  int best_b = 1;
  for (int b = sk::kMaxBoxesPerStage; b >= 1; --b) {
    if (b > 1 && nkb % b) continue;  // whole stages: a box never reads past the slice
    const int need = std::min(3, (nkb + b - 1) / b);
    if (bytes(need, b) <= budget) {
      best_b = b;
      break;
    }
  }
  if (const int bv = env_int("SK_BPS", 1, sk::kMaxBoxesPerStage)) best_b = bv;
  int st = 1;
  while (st < sk::kMaxStages && bytes(st + 1, best_b) <= budget) ++st;
  if (const int sv = env_int("SK_STAGES", 1, sk::kMaxStages)) st = sv;
  const int nst = (nkb + best_b - 1) / best_b;
  *stages = st < nst ? st : nst;
  *bps = best_b;
}

// The weight stream is the whole cost; what sets its rate is the number of
// bytes in flight from HBM (tens of MB GPU-wide) and the size of each copy.
// Long K (>= 2048): full 128-row tiles, and the largest split count S that
// keeps every CTA resident at two per SM (tiles x S <= 2 x SMs, clusters
// schedulable) with at least 8 K blocks per CTA. When that plan would leave
// more than half the SMs idle (few output rows), 64-row tiles instead, with
// the largest S <= 4 at one CTA per SM: the same CTAs read half the operand
// bytes per MMA and exchange across fewer ranks ([1024, 4096] at M = 16:
// 4.2 against 4.6 us per dependent call). Short K: no split, one wave of
// CTAs one per SM with the rows spread evenly (the 64-row MMA for up to 64
// rows). The ring takes all the shared memory the residency allows. A
// requested split count is honoured.
GemmPlan plan_gemm(int n, int k, int splits_req, int device, int sm_count) {
  GemmPlan p{0, 0, 0, 1};
  const int nkb_total = k / sk::kBlockK;
  auto fits = [&](int s, int tiles, int per_sm, int h) {
    if (tiles * s > per_sm * sm_count) return false;
    if (s == 1) return true;
    const int c = sk::gemm_max_clusters(device, s, per_sm, h);
    return c <= 0 || tiles <= c;
  };
  if (splits_req) {
    p.splits = splits_req;
    const int cap = 2 * sm_count / splits_req;
    int h = (n + (cap > 0 ? cap : 1) - 1) / (cap > 0 ? cap : 1);
    p.h = h < 16 ? 16 : (h > sk::kMmaM ? sk::kMmaM : h);
    if (k >= 2048) p.h = sk::kMmaM;
  } else if (k >= 2048) {
    p.h = sk::kMmaM;
    const int tiles = (n + p.h - 1) / p.h;
    p.splits = 1;
    for (int s = 2; s <= 16; s *= 2) {
      if (nkb_total % s || nkb_total / s < 8) break;
      if (!fits(s, tiles, 2, p.h)) break;
      p.splits = s;
    }
    if (2 * tiles * p.splits <= sm_count) {
      p.h = 64;
      const int tiles64 = (n + p.h - 1) / p.h;
      p.splits = 1;
      for (int s = 2; s <= 4; s *= 2) {
        if (nkb_total % s || nkb_total / s < 8) break;
        if (!fits(s, tiles64, 1, p.h)) break;
        p.splits = s;
      }
    }
  } else {
    p.splits = 1;
    int h = (n + sm_count - 1) / sm_count;
    p.h = h < 16 ? 16 : (h > sk::kMmaM ? sk::kMmaM : h);
  }
  if (const int hv = env_int("SK_TILE_ROWS", 16, sk::kMmaM)) p.h = hv;
  p.h = (p.h + 7) / 8 * 8;  // whole 8-row swizzle atoms per 64-column block
  const int tiles = (n + p.h - 1) / p.h;
  const size_t budget = tiles * p.splits <= sm_count ? sk::kOnePerSmSmem : sk::kTwoPerSmSmem;
  choose_ring(nkb_total / p.splits, budget,
              [&](int st, int b) { return sk::gemm_smem_bytes(p.h, st, b, p.splits); }, &p.stages, &p.bps);
  return p;
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

sk_status launch_status(cudaError_t e, const char *what) {
  if (e != cudaSuccess) return fail(SK_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  return ok();
}

// The weight of the GEMM this host thread enqueues after the next one
// (sk_gemm_prefetch_next); consumed by the next GEMM enqueue. t_prefetched:
// the weight whose first stages the last GEMM enqueue started towards L2.
struct PrefetchHint {
  const void *w = nullptr;
  int n = 0, k = 0;
  bool operator==(const PrefetchHint &o) const { return w == o.w && n == o.n && k == o.k; }
};
thread_local PrefetchHint t_prefetch;
thread_local PrefetchHint t_prefetched;

// Stages of the next GEMM's slice that each of its CTAs has started towards
// L2 by the previous GEMM: about 448 KiB per CTA, at most 64 MiB in all
// (measured best on the decode chain, where this GEMM's own look-ahead is then
// left out; more slows the norm kernels between the GEMMs). SK_PF_STAGES
// overrides (0: none).
int prefetch_stages(const GemmPlan &next, int tiles) {
  const char *v = std::getenv("SK_PF_STAGES");
  if (v && *v) {
    const int n = std::atoi(v);
    return n < 0 ? 0 : (n > 64 ? 64 : n);
  }
  const long stage_w = static_cast<long>(next.bps) * next.h * 128;
  const long per_cta = (448L * 1024 + stage_w - 1) / stage_w;
  const long cap = (64L << 20) / (stage_w * tiles * next.splits);
  return static_cast<int>(std::max(1L, std::min(per_cta, cap)));
}

// Validated GEMM enqueue shared by the three GEMM entry points.
sk_status enqueue_gemm(const void *x, const void *w, void *y, int m, int n, int k, int splits,
                       void *stream, const sk::DeviceInfo &info, bool x_ready = false) {
  const PrefetchHint hint = t_prefetch;
  // this GEMM's first weight stages were started by the previous one: no
  // look-ahead of its own
  const bool warmed = t_prefetched.w && t_prefetched == PrefetchHint{w, n, k};
  t_prefetch = PrefetchHint{};
  t_prefetched = PrefetchHint{};
  int dev = 0;
  cudaGetDevice(&dev);
  const GemmPlan plan = plan_gemm(n, k, splits, dev, info.sm_count);
  if (plan.splits == 0)
    return fail(SK_ERR_UNSUPPORTED, "no GEMM launch for n=%d, k=%d, splits=%d", n, k, splits);
  CUtensorMap tw, tx;
  sk_status st;
  if ((st = make_map(&tw, w, n, k, plan.h, plan.bps)) != SK_OK) return st;
  if ((st = make_map(&tx, x, m, k, sk::kTokTile, plan.bps)) != SK_OK) return st;
  sk::GemmPrefetch pf;
  const sk::GemmPrefetch *pfp = nullptr;
  if (hint.w) {
    const GemmPlan np = plan_gemm(hint.n, hint.k, 0, dev, info.sm_count);
    pf.stages = np.splits ? prefetch_stages(np, (hint.n + np.h - 1) / np.h) : 0;
    if (pf.stages > 0) {
      if ((st = make_map(&pf.map, hint.w, hint.n, hint.k, np.h, np.bps)) != SK_OK) return st;
      pf.h = np.h;
      pf.nkb = hint.k / sk::kBlockK / np.splits;
      pf.bps = np.bps;
      pf.tiles = (hint.n + np.h - 1) / np.h;
      pf.splits = np.splits;
      pfp = &pf;
    }
  }
  st = launch_status(sk::launch_gemm(tw, tx, static_cast<uint16_t *>(y), m, n, k, plan.splits,
                                     plan.h, plan.stages, plan.bps, as_stream(stream),
                                     pdl_enabled(), pfp, warmed ? 0 : -1, x_ready),
                     "gemm");
  if (st == SK_OK && pfp) t_prefetched = hint;
  return st;
}

sk_status check_ptrs16(const char *names, std::initializer_list<const void *> ps) {
  int i = 0;
  for (const void *p : ps) {
    if (!p) return fail(SK_ERR_INVALID_ARG, "null pointer (argument %d of %s)", i, names);
    if (!aligned16(p))
      return fail(SK_ERR_INVALID_ARG, "pointer %p (argument %d of %s) is not 16-byte aligned", p, i,
                  names);
    ++i;
  }
  return SK_OK;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// ------------------------------------------------- weight-only NVFP4 GEMM
sk_status check_nvfp4w_shape(int m, int n, int k, int splits) {
  if (m < 1 || m > SK_MAX_M)
    return fail(SK_ERR_INVALID_ARG, "m=%d: needs 1 <= m <= %d token rows", m, SK_MAX_M);
  if (n <= 0 || n % 16)
    return fail(SK_ERR_INVALID_ARG, "n=%d: needs a positive multiple of 16 output features", n);
  if (k <= 0 || k % sk::kW4BlockK)
    return fail(SK_ERR_INVALID_ARG, "k=%d: needs a positive multiple of %d", k, sk::kW4BlockK);
  if (splits != 0 && splits != 1 && splits != 2 && splits != 4 && splits != 8 && splits != 16)
    return fail(SK_ERR_UNSUPPORTED, "unsupported split count %d (0, 1, 2, 4, 8 or 16)", splits);
  if (splits > 0 && k % (sk::kW4BlockK * splits))
    return fail(SK_ERR_UNSUPPORTED, "K=%d does not split into %d slices of whole %d-wide blocks", k,
                splits, sk::kW4BlockK);
  return SK_OK;
}

// Split count and ring depth of the weight-only NVFP4 GEMM. One CTA per SM
// (each takes all of its SM's tensor memory): the largest S that keeps the
// grid within one wave of resident clusters with at least two K blocks per
// CTA; the ring as deep as shared memory allows.
struct W4Plan {
  int splits, stages;
};

W4Plan plan_nvfp4w(int n, int k, int splits_req, int device, int sm_count) {
  W4Plan p{1, 1};
  const int tiles = (n + sk::kW4Rows - 1) / sk::kW4Rows;
  const int nblk = k / sk::kW4BlockK;
  if (splits_req) {
    p.splits = splits_req;
  } else {
    for (int s = 2; s <= 16; s *= 2) {
      if (nblk % s || nblk / s < 2) break;
      if (tiles * s > sm_count) break;
      const int c = sk::w4_max_clusters(device, s);
      if (c > 0 && tiles > c) break;
      p.splits = s;
    }
  }
  const int per = nblk / p.splits;
  int st = 1;
  while (st < sk::kW4MaxStages && sk::w4_smem_bytes(st + 1, p.splits) <= sk::kOnePerSmSmem) ++st;
  if (const int sv = env_int("SK_STAGES", 1, sk::kW4MaxStages)) st = sv;
  p.stages = st < per ? st : per;
  return p;
}

}  // namespace

sk_status sk::report_error(sk_status st, const char *msg) { return fail(st, "%s", msg); }

sk_status sk::checked_device(sk::DeviceInfo *info, int *device) {
  sk_status st = current_device(info);
  if (st != SK_OK) return st;
  cudaGetDevice(device);
  return SK_OK;
}

bool sk::pdl_on() { return pdl_enabled(); }

extern "C" {

const char *sk_last_error(void) { return t_last_error.c_str(); }

int sk_version(void) { return SK_VERSION; }

sk_status sk_gemm_supported(int m, int n, int k, int splits) {
  sk_status st = check_gemm_shape(m, n, k, splits);
  return st == SK_OK ? ok() : st;
}

int sk_gemm_splits(int m, int n, int k, int splits) {
  if (check_gemm_shape(m, n, k, splits) != SK_OK) return 0;
  if (splits) return splits;
  sk::DeviceInfo info;
  if (current_device(&info) != SK_OK) return 0;
  int dev = 0;
  cudaGetDevice(&dev);
  ok();
  return plan_gemm(n, k, 0, dev, info.sm_count).splits;
}

sk_status sk_gemm_bf16(const void *x, const void *w, void *y, int m, int n, int k, int splits,
                       void *stream) {
  sk_status st;
  if ((st = check_gemm_shape(m, n, k, splits)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_bf16(x, w, y)", {x, w, y})) != SK_OK) return st;
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  return enqueue_gemm(x, w, y, m, n, k, splits, stream, info);
}

sk_status sk_gemm_bf16_ex(const void *x, const void *w, void *y, int m, int n, int k, int splits,
                          unsigned flags, void *stream) {
  if (flags & ~SK_GEMM_X_READY) return fail(SK_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  sk_status st;
  if ((st = check_gemm_shape(m, n, k, splits)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_bf16_ex(x, w, y)", {x, w, y})) != SK_OK) return st;
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  return enqueue_gemm(x, w, y, m, n, k, splits, stream, info, (flags & SK_GEMM_X_READY) != 0);
}

sk_status sk_gemm_prefetch_next(const void *w_next, int n_next, int k_next) {
  if (!w_next) {
    t_prefetch = PrefetchHint{};
    return ok();
  }
  sk_status st;
  if ((st = check_gemm_shape(1, n_next, k_next, 0)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_prefetch_next(w_next)", {w_next})) != SK_OK) return st;
  t_prefetch = PrefetchHint{w_next, n_next, k_next};
  return ok();
}

static sk_status check_norm_quant(int m, int n) {
  if (m < 1 || m > SK_MAX_M)
    return fail(SK_ERR_INVALID_ARG, "m=%d: needs 1 <= m <= %d token rows", m, SK_MAX_M);
  if (n < 16 || n % 16 || n > 16384)
    return fail(SK_ERR_INVALID_ARG, "n=%d: needs a multiple of 16 in [16, 16384]", n);
  return SK_OK;
}

sk_status sk_rmsnorm_nvfp4(const void *y, const void *norm_w, float eps, float gain_center,
                           const float *global_scale, uint8_t *a, uint8_t *a_sf, void *z_out,
                           int m, int n, void *stream) {
  sk_status st;
  if ((st = check_norm_quant(m, n)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_rmsnorm_nvfp4(y, norm_w, a)", {y, norm_w, a})) != SK_OK) return st;
  if (!global_scale || (reinterpret_cast<uintptr_t>(global_scale) & 3))
    return fail(SK_ERR_INVALID_ARG, "global_scale must be a 4-byte aligned device FP32 [1]");
  if (!a_sf) return fail(SK_ERR_INVALID_ARG, "a_sf is null");
  if (z_out && !aligned16(z_out)) return fail(SK_ERR_INVALID_ARG, "z_out is not 16-byte aligned");
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  return launch_status(
      sk::launch_rmsnorm_nvfp4(static_cast<const uint16_t *>(y), static_cast<const uint16_t *>(norm_w),
                               eps, gain_center, global_scale, a, a_sf,
                               static_cast<uint16_t *>(z_out), m, n, as_stream(stream),
                               pdl_enabled()),
      "rmsnorm_nvfp4");
}

size_t sk_gemm_rmsnorm_nvfp4_workspace(int m, int n) {
  if (m <= 0 || n <= 0) return 0;
  return round256(static_cast<size_t>(m) * n * 2);
}

sk_status sk_gemm_rmsnorm_nvfp4(const void *x, const void *w, const void *norm_w, float eps,
                                float gain_center, const float *global_scale, uint8_t *a,
                                uint8_t *a_sf, void *z_out, void *workspace,
                                size_t workspace_bytes, int m, int n, int k, int splits,
                                void *stream) {
  sk_status st;
  if ((st = check_gemm_shape(m, n, k, splits)) != SK_OK) return st;
  if ((st = check_norm_quant(m, n)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_rmsnorm_nvfp4(x, w, norm_w, a, workspace)",
                         {x, w, norm_w, a, workspace})) != SK_OK)
    return st;
  if (!global_scale || (reinterpret_cast<uintptr_t>(global_scale) & 3))
    return fail(SK_ERR_INVALID_ARG, "global_scale must be a 4-byte aligned device FP32 [1]");
  if (!a_sf) return fail(SK_ERR_INVALID_ARG, "a_sf is null");
  if (z_out && !aligned16(z_out)) return fail(SK_ERR_INVALID_ARG, "z_out is not 16-byte aligned");
  if (workspace_bytes < sk_gemm_rmsnorm_nvfp4_workspace(m, n))
    return fail(SK_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes,
                sk_gemm_rmsnorm_nvfp4_workspace(m, n));
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  if ((st = enqueue_gemm(x, w, workspace, m, n, k, splits, stream, info)) != SK_OK) return st;
  return launch_status(
      sk::launch_rmsnorm_nvfp4(static_cast<const uint16_t *>(workspace),
                               static_cast<const uint16_t *>(norm_w), eps, gain_center,
                               global_scale, a, a_sf, static_cast<uint16_t *>(z_out), m, n,
                               as_stream(stream), pdl_enabled()),
      "rmsnorm_nvfp4");
}

sk_status sk_rmsnorm_bf16(const void *y, const void *norm_w, float eps, float gain_center, void *z,
                          int m, int n, void *stream) {
  sk_status st;
  if ((st = check_norm_quant(m, n)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_rmsnorm_bf16(y, norm_w, z)", {y, norm_w, z})) != SK_OK) return st;
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  return launch_status(
      sk::launch_rmsnorm_nvfp4(static_cast<const uint16_t *>(y), static_cast<const uint16_t *>(norm_w),
                               eps, gain_center, nullptr, nullptr, nullptr,
                               static_cast<uint16_t *>(z), m, n, as_stream(stream), pdl_enabled()),
      "rmsnorm_bf16");
}

sk_status sk_gemm_rmsnorm_bf16(const void *x, const void *w, const void *norm_w, float eps,
                               float gain_center, void *z, void *workspace,
                               size_t workspace_bytes, int m, int n, int k, int splits,
                               void *stream) {
  sk_status st;
  if ((st = check_gemm_shape(m, n, k, splits)) != SK_OK) return st;
  if ((st = check_norm_quant(m, n)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_rmsnorm_bf16(x, w, norm_w, z, workspace)",
                         {x, w, norm_w, z, workspace})) != SK_OK)
    return st;
  if (workspace_bytes < sk_gemm_rmsnorm_nvfp4_workspace(m, n))
    return fail(SK_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes,
                sk_gemm_rmsnorm_nvfp4_workspace(m, n));
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  if ((st = enqueue_gemm(x, w, workspace, m, n, k, splits, stream, info)) != SK_OK) return st;
  return launch_status(
      sk::launch_rmsnorm_nvfp4(static_cast<const uint16_t *>(workspace),
                               static_cast<const uint16_t *>(norm_w), eps, gain_center, nullptr,
                               nullptr, nullptr, static_cast<uint16_t *>(z), m, n,
                               as_stream(stream), pdl_enabled()),
      "rmsnorm_bf16");
}

sk_status sk_nvfp4_quantize(const void *z, const float *global_scale, uint8_t *a, uint8_t *a_sf,
                            int m, int n, void *stream) {
  sk_status st;
  if (m < 1 || m > 65535) return fail(SK_ERR_INVALID_ARG, "m=%d: needs 1 <= m <= 65535", m);
  if (n < 16 || n % 16) return fail(SK_ERR_INVALID_ARG, "n=%d: needs a positive multiple of 16", n);
  if ((st = check_ptrs16("sk_nvfp4_quantize(z, a)", {z, a})) != SK_OK) return st;
  if (!global_scale || (reinterpret_cast<uintptr_t>(global_scale) & 3))
    return fail(SK_ERR_INVALID_ARG, "global_scale must be a 4-byte aligned device FP32 [1]");
  if (!a_sf) return fail(SK_ERR_INVALID_ARG, "a_sf is null");
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  return launch_status(sk::launch_nvfp4_quantize(static_cast<const uint16_t *>(z), global_scale, a,
                                                 a_sf, m, n, as_stream(stream), pdl_enabled()),
                       "nvfp4_quantize");
}

static sk_status check_dual(const void *partial, const float *resid, const void *post_w,
                            const void *beta, const void *pre_w, const void *out, int m, int h) {
  if (m < 1 || m > SK_MAX_M)
    return fail(SK_ERR_INVALID_ARG, "m=%d: needs 1 <= m <= %d token rows", m, SK_MAX_M);
  if (h < 8 || h % 8 || h > 8192)
    return fail(SK_ERR_INVALID_ARG, "h=%d: needs a multiple of 8 in [8, 8192]", h);
  sk_status st = check_ptrs16("sk_dual_norm_residual(partial, resid, beta, pre_w, out)",
                              {partial, resid, beta, pre_w, out});
  if (st != SK_OK) return st;
  if (post_w && !aligned16(post_w)) return fail(SK_ERR_INVALID_ARG, "post_w is not 16-byte aligned");
  return SK_OK;
}

sk_status sk_dual_norm_residual(const void *partial, float *resid, const void *post_w, float alpha,
                                const void *beta, const void *pre_w, void *out, float eps_post,
                                float eps_pre, float gc_post, float gc_pre, int m, int h,
                                void *stream) {
  sk_status st;
  if ((st = check_dual(partial, resid, post_w, beta, pre_w, out, m, h)) != SK_OK) return st;
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  return launch_status(
      sk::launch_dual_norm(static_cast<const uint16_t *>(partial), resid,
                           static_cast<const uint16_t *>(post_w), alpha,
                           static_cast<const uint16_t *>(beta), static_cast<const uint16_t *>(pre_w),
                           static_cast<uint16_t *>(out), eps_post, eps_pre, gc_post, gc_pre, m, h,
                           as_stream(stream), pdl_enabled()),
      "dual_norm");
}

size_t sk_gemm_dual_norm_workspace(int m, int n) {
  if (m <= 0 || n <= 0) return 0;
  return round256(static_cast<size_t>(m) * n * 2);
}

sk_status sk_gemm_dual_norm(const void *x, const void *w, float *resid, const void *post_w,
                            float alpha, const void *beta, const void *pre_w, void *out,
                            float eps_post, float eps_pre, float gc_post, float gc_pre,
                            void *workspace, size_t workspace_bytes, int m, int n, int k,
                            int splits, void *stream) {
  sk_status st;
  if ((st = check_gemm_shape(m, n, k, splits)) != SK_OK) return st;
  if ((st = check_dual(workspace, resid, post_w, beta, pre_w, out, m, n)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_dual_norm(x, w)", {x, w})) != SK_OK) return st;
  if (workspace_bytes < sk_gemm_dual_norm_workspace(m, n))
    return fail(SK_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes,
                sk_gemm_dual_norm_workspace(m, n));
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  if ((st = enqueue_gemm(x, w, workspace, m, n, k, splits, stream, info)) != SK_OK) return st;
  return launch_status(
      sk::launch_dual_norm(static_cast<const uint16_t *>(workspace), resid,
                           static_cast<const uint16_t *>(post_w), alpha,
                           static_cast<const uint16_t *>(beta), static_cast<const uint16_t *>(pre_w),
                           static_cast<uint16_t *>(out), eps_post, eps_pre, gc_post, gc_pre, m, n,
                           as_stream(stream), pdl_enabled()),
      "dual_norm");
}

sk_status sk_gemm_nvfp4w_supported(int m, int n, int k, int splits) {
  sk_status st = check_nvfp4w_shape(m, n, k, splits);
  return st == SK_OK ? ok() : st;
}

int sk_gemm_nvfp4w_splits(int m, int n, int k, int splits) {
  if (check_nvfp4w_shape(m, n, k, splits) != SK_OK) return 0;
  if (splits) return splits;
  sk::DeviceInfo info;
  if (current_device(&info) != SK_OK) return 0;
  int dev = 0;
  cudaGetDevice(&dev);
  ok();
  return plan_nvfp4w(n, k, 0, dev, info.sm_count).splits;
}

sk_status sk_gemm_nvfp4w_bf16(const void *x, const uint8_t *wq, const uint8_t *wsf,
                              const float *w_scale, void *y, int m, int n, int k, int splits,
                              void *stream) {
  sk_status st;
  if ((st = check_nvfp4w_shape(m, n, k, splits)) != SK_OK) return st;
  if ((st = check_ptrs16("sk_gemm_nvfp4w_bf16(x, wq, wsf, y)", {x, wq, wsf, y})) != SK_OK) return st;
  if (!w_scale || (reinterpret_cast<uintptr_t>(w_scale) & 3))
    return fail(SK_ERR_INVALID_ARG, "w_scale must be a 4-byte aligned device FP32 [1]");
  sk::DeviceInfo info;
  if ((st = current_device(&info)) != SK_OK) return st;
  int dev = 0;
  cudaGetDevice(&dev);
  const W4Plan plan = plan_nvfp4w(n, k, splits, dev, info.sm_count);
  CUtensorMap tq, tsf, tx;
  if ((st = make_byte_map(&tq, wq, n, k / 2, 128, sk::kW4Rows, true)) != SK_OK) return st;
  if ((st = make_byte_map(&tsf, wsf, n, k / 16, 16, sk::kW4Rows, false)) != SK_OK) return st;
  if ((st = make_map(&tx, x, m, k, sk::kTokTile, sk::kW4BlockK / sk::kBlockK)) != SK_OK) return st;
  // about 256 KiB of each CTA's code and scale blocks beyond the ring start
  // towards L2 before the dependency wait
  const int l2_ahead = (256 * 1024 + sk::kW4CodeBytes + sk::kW4ScaleBytes - 1) /
                       (sk::kW4CodeBytes + sk::kW4ScaleBytes);
  return launch_status(sk::launch_gemm_nvfp4w(tq, tsf, tx, w_scale, static_cast<uint16_t *>(y), m,
                                              n, k, plan.splits, plan.stages, l2_ahead,
                                              as_stream(stream), pdl_enabled()),
                       "gemm_nvfp4w");
}

sk_status sk_wait_probe(unsigned limit_us, void *stream) {
  if (limit_us < 1 || limit_us > 100000)
    return fail(SK_ERR_INVALID_ARG, "limit_us=%u: needs 1 <= limit_us <= 100000", limit_us);
  sk::DeviceInfo info;
  sk_status st;
  if ((st = current_device(&info)) != SK_OK) return st;
  return launch_status(sk::launch_wait_probe(static_cast<uint64_t>(limit_us) * 1000, as_stream(stream)),
                       "wait_probe");
}

sk_status sk_device_status(uint32_t *out, int clear) {
  if (!out) return fail(SK_ERR_INVALID_ARG, "out is null");
  sk::DeviceInfo info;
  sk_status st;
  if ((st = current_device(&info)) != SK_OK) return st;
  cudaError_t e = sk::read_device_status(out, clear != 0);
  if (e != cudaSuccess) return fail(SK_ERR_CUDA, "device status read failed: %s", cudaGetErrorString(e));
  return ok();
}

sk_status sk_convert_probe(int kind, const void *in, void *out, int n, void *stream) {
  if (kind < 0 || kind > 3) return fail(SK_ERR_INVALID_ARG, "kind=%d: needs 0..3", kind);
  if (n < 0) return fail(SK_ERR_INVALID_ARG, "n=%d < 0", n);
  if (n == 0) return ok();
  if (!in || !out) return fail(SK_ERR_INVALID_ARG, "null pointer");
  sk::DeviceInfo info;
  sk_status st;
  if ((st = current_device(&info)) != SK_OK) return st;
  return launch_status(sk::launch_convert_probe(kind, in, out, n, as_stream(stream)), "convert_probe");
}

}  // extern "C"
