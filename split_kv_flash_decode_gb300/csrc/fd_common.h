// Internal definitions shared by the host planner (fd_api.cpp) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>              // CUtensorMap
#include <cuda_runtime_api.h>

#include "../../include/fd.h"

#if defined(__CUDACC__)
#define FD_HD __host__ __device__ __forceinline__
#else
#define FD_HD inline
#endif

namespace fd {

// Tokens per pipeline stage (rows of K and of V moved by one pair of TMA loads).
constexpr int kTile = 32;
// Consumer warps per CTA; one more warp issues the TMA loads.
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// Stages of the shared-memory ring per head dimension.
FD_HD constexpr int stages_for(int d) { return d == 128 ? 6 : 8; }

// Dynamic shared memory of one CTA: the K/V ring plus the mbarriers.
FD_HD constexpr size_t smem_bytes_for(int d) {
  return (size_t)stages_for(d) * 2 * kTile * d * 2 + 1024;
}

// Status word values written by the kernels (the host maps them to fd_status).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusCounter = 2u;

// Kernel parameters (passed by value as a __grid_constant__ struct; < 4 KB).
struct Params {
  CUtensorMap tm_k;  // 3-D view of K: (d, Hkv, N), box (d, 1, kTile)
  CUtensorMap tm_v;  // same for V
  const void* q;     // [B, Hq, d]
  void* out;         // [B, Hq, d]
  float* lse;        // [B, Hq] or nullptr
  float* part_o;     // [P, d]
  float* part_m;     // [P]   (log2-domain maxima of the scaled logits)
  float* part_l;     // [P]
  uint32_t* counters;  // [B * Hkv]
  uint32_t* status;    // 1 word
  float scale_log2;    // log2(e) / sqrt(d)
  int32_t B, Hq, Hkv, C;
  int32_t cu[FD_MAX_BATCH + 1];         // token prefix sums
  int32_t unit_base[FD_MAX_BATCH + 1];  // prefix sums of Hkv * W_b * C (CTA index base)
  uint16_t wseg[FD_MAX_BATCH];          // W_b
};
static_assert(sizeof(Params) <= 4096, "kernel parameters must stay within 4 KB");

// Token range of partial `slot` of a sequence of length L split into W segments
// of ceil(L/W) tokens, each cut into C chunks of ceil(n/C) tokens.
FD_HD void chunk_range(int L, int W, int C, int slot, int* t0, int* t1) {
  const int w = slot / C, c = slot - (slot / C) * C;
  const int64_t S = L > 0 ? ((int64_t)L + W - 1) / W : 0;
  int64_t sb = (int64_t)w * S;
  if (sb > L) sb = L;
  int64_t se = sb + S;
  if (se > L) se = L;
  const int64_t n = se - sb;
  const int64_t cl = (n + C - 1) / C;
  int64_t a = (int64_t)c * cl, e = (int64_t)(c + 1) * cl;
  if (a > n) a = n;
  if (e > n) e = n;
  *t0 = (int)(sb + a);
  *t1 = (int)(sb + e);
}

// Launchers defined in the per-dtype kernel translation units.
// mode 0: fused split + last-arriver combine; 1: split only (partials); 2: combine only.
cudaError_t launch_f16(const Params& p, int d, int G, int mode, int grid, cudaStream_t s);
cudaError_t launch_bf16(const Params& p, int d, int G, int mode, int grid, cudaStream_t s);

}  // namespace fd
