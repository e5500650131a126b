// Internal plan layout shared by the host translation units of the library.
#pragma once

#include "fd_common.h"

struct fd_plan_s {
  int B, Hq, Hkv, d, G, dtype;
  uint32_t flags;
  int C;
  int path;       // fd::kPathFfma or fd::kPathMma
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
