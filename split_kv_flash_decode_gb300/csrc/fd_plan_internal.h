// Internal plan layout shared by the host translation units of the library.
#pragma once

#include "fd_common.h"

struct fd_plan_s {
  int B, Hq, Hkv, d, G, dtype;
  uint32_t flags;
  int C;
  int path;  // fd::kPathFfma or fd::kPathMma
  int num_sms;
  int max_partials;
  int64_t n_tokens;
  int64_t total_partials;
  int ctas;
  size_t off_counters, off_flags, off_part, ws_bytes;
  fd::Params params;  // pointers filled per call; arrays and scalars filled by fd_plan
};

namespace fd {
// Encode the 3-D TMA view (d, Hkv, N) of a [N, Hkv, d] K or V tensor at `base`.
int encode_kv_map(CUtensorMap* map, const void* base, const fd_plan_s* pl);
}  // namespace fd
