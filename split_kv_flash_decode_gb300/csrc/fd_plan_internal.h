// Internal plan layout shared by the host translation units of the library.
#pragma once

#include "fd_common.h"

struct fd_plan_s {
  int B, Hq, Hkv, d, G, dtype;
  uint32_t flags;
  int C;
  int path;       // fd::kPathFfma, kPathMma, kPathMmaKv8 or kPathUmma
  int page_size;  // 0: contiguous K/V; else tokens per page of a paged cache
  int max_pages;  // max_b ceil(L_b / page_size) (paged plans)
  int num_sms;
  int max_partials;
  int64_t n_tokens;
  int64_t total_partials;
  int ctas;
  size_t off_counters, off_flags, off_part, ws_bytes;
  fd::Params params;  // pointers filled per call; arrays and scalars filled by fd_plan
};

namespace fd {
// Encode the 3-D TMA view (d, Hkv, rows) of a [rows, Hkv, d] K or V tensor (or page
// pool) at `base`; one box is `box_rows` token rows of one head.
int encode_kv_map(CUtensorMap* map, const void* base, int64_t rows, int box_rows,
                  const fd_plan_s* pl);
}  // namespace fd

namespace fd {
// Kernel mode of a one-launch decode: fine-grained waits (3), every partial of a pair
// in one cluster (6), or the last-arriver combine (0).
inline int fused_mode(const fd_plan_s* pl) {
  return (pl->flags & FD_PLAN_WAITS) ? 3 : (pl->flags & FD_PLAN_CLUSTER_COMBINE) ? 6 : 0;
}
// fd_status of a failed launch: a grid that cannot be co-resident (cooperative
// launch) or a cluster the device cannot place is unsupported; anything else is a
// CUDA failure.
inline int launch_status(cudaError_t err) {
  return (err == cudaErrorCooperativeLaunchTooLarge || err == cudaErrorInvalidClusterSize)
             ? FD_ERR_UNSUPPORTED
             : FD_ERR_CUDA;
}
// One kernel launch of the plan's consumer path and dtype (mode as listed above the
// launcher declarations).
inline cudaError_t launch_plan(const fd_plan_s* pl, const Params& p, int mode, int grid,
                               cudaStream_t s) {
  const bool pdl = !(pl->flags & FD_PLAN_NO_PDL);
  if (pl->path == kPathUmma)
    return pl->dtype == FD_BF16 ? launch_umma_bf16(p, pl->d, pl->G, mode, pdl, grid, s)
                                : launch_umma_f16(p, pl->d, pl->G, mode, pdl, grid, s);
  if (pl->path == kPathFfma)
    return pl->dtype == FD_BF16 ? launch_bf16_ffma(p, pl->d, pl->G, mode, pdl, grid, s)
                                : launch_f16_ffma(p, pl->d, pl->G, mode, pdl, grid, s);
  return pl->dtype == FD_BF16 ? launch_bf16_mma(p, pl->d, pl->G, pl->path, mode, pdl, grid, s)
                              : launch_f16_mma(p, pl->d, pl->G, pl->path, mode, pdl, grid, s);
}
}  // namespace fd
