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

// GEMM tiling: each CTA owns kTileN consecutive weight rows (output features)
// and one K slice; the tensor-core instruction is M = kTileN weight rows by
// N = kTokTile token columns (rows of x beyond m are zero-filled by the copy
// engine), K = 16 per instruction, kBlockK per pipeline stage.
constexpr int kTileN = 128;
constexpr int kTokTile = 16;
constexpr int kBlockK = 64;
constexpr int kStageWBytes = kTileN * kBlockK * 2;   // 16 KiB weight box
constexpr int kStageXBytes = kTokTile * kBlockK * 2; // 2 KiB activation box
constexpr int kMaxStages = 12;

struct DeviceInfo {
  int sm_count = 0;
  int major = 0, minor = 0;
  size_t max_smem_optin = 0;
};

// Per-device properties and one-time kernel attribute set-up for the current
// device. Returns cudaSuccess or the first error.
cudaError_t device_setup(int device, DeviceInfo *info);

size_t gemm_smem_bytes(int stages);

// Launches the split-K GEMM: grid (ceil(n / kTileN), splits), cluster
// (1, splits, 1); `stages` pipeline stages per CTA.
cudaError_t launch_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, uint16_t *y, int m,
                        int n, int k, int splits, int stages, cudaStream_t stream, bool pdl);

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

cudaError_t read_device_status(uint32_t *out, bool clear);

}  // namespace sk
