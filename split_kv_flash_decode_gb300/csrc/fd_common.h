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

// Consumer warps per CTA; one more warp issues the TMA loads.
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// Two consumer paths.  FFMA: CUDA-core dot products, unswizzled [tile][d] rows.
// MMA: mma.sync m16n8k16 with tokens on M and the GQA heads on N, K/V staged as
// 64-column half-tiles with the 128-byte TMA swizzle (conflict-free ldmatrix).
// KV8: the MMA path over an FP8 (E4M3) cache, d = 128 only.  K/V land in the ring
// as 128-byte swizzled rows of bytes; every thread loads its mma fragments from
// there directly and widens them to f16 with integer ops.
constexpr int kPathFfma = 0;
constexpr int kPathMma = 1;
constexpr int kPathMmaKv8 = 2;

FD_HD constexpr bool is_mma(int path) { return path != kPathFfma; }
// Bytes per stored K/V element.
FD_HD constexpr int kv_elem_bytes(int path) { return path == kPathMmaKv8 ? 1 : 2; }
// Tokens per pipeline stage.
FD_HD constexpr int tile_for(int path) { return is_mma(path) ? 64 : 32; }
// Columns (elements) of one TMA box row: 128-byte swizzled rows on the MMA paths.
FD_HD constexpr int box_cols_for(int path, int d) {
  return path == kPathMma ? 64 : path == kPathMmaKv8 ? 128 : d;
}
// K/V tiles per CTA that the split kernel prefetches into L2 before it waits for
// the previous kernel in the stream (4 measured best for fp16 and fp8 caches at
// 32K and 128K tokens; 2 and 8 were slower).
constexpr int kL2PrefetchTiles = 4;
// The K/V ring, 96 KB on every path: slots of one tile of K rows followed by the
// tile of V rows of one KV head.  (At d = 64 the ring used to be 64 KB; 96 KB is
// 14% faster at 32K tokens.  A 112 KB ring, the most two CTAs per SM can hold,
// was slower on every path, and so were separate K and V slots with their own
// barriers on the multi-wave and FP8 cases.)
constexpr int kRingBytes = 96 * 1024;
FD_HD constexpr int slot_bytes_for(int path, int d) { return 2 * tile_for(path) * d * kv_elem_bytes(path); }
FD_HD constexpr int ring_slots_for(int path, int d) { return kRingBytes / slot_bytes_for(path, d); }
// Bytes of the K/V ring (also the scratch the combine reuses).
FD_HD constexpr size_t ring_bytes_for(int path, int d) {
  return (size_t)ring_slots_for(path, d) * slot_bytes_for(path, d);
}
// Bytes after the ring: 2 mbarriers per slot, the combine's mbarrier, two flags,
// and up to 1 KB of slack for aligning the ring to 1024 bytes.
constexpr int kRingMetaBytes = 2048;
// Dynamic shared memory of one CTA: the ring and its metadata.
FD_HD constexpr size_t smem_bytes_for(int path, int d) { return ring_bytes_for(path, d) + kRingMetaBytes; }
// Floats per partial record: O[0..d), m, l and two pad words (16-byte records).
FD_HD constexpr int record_floats(int d) { return d + 4; }

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
  float* part;       // [P, d + 4] records: O[0..d), m, l, 0, 0 (m in the log2 domain)
  uint32_t* counters;  // [B * Hkv]
  uint32_t* flags;     // [CTAs] per-partial ready flags (fine-grained-waits variant)
  uint32_t* status;    // 1 word
  int32_t drop_flag;   // test hook: partial slot 1 of (b=0, kvh=0) never sets its flag
  // Paged KV cache: K/V rows of sequence b, token t live at pool row
  // block_table[b * bt_stride + (t >> page_shift)] * page_size + (t & (page_size - 1)).
  const int32_t* block_table;  // nullptr: contiguous [N, Hkv, d] layout
  int32_t bt_stride;
  int32_t page_shift;
  int32_t box_rows;    // token rows per TMA box (the tile, or one page when pages are smaller)
  int32_t align;       // segment / chunk boundaries are multiples of this many tokens
  int32_t prefetch_ctas;  // CTAs [0, prefetch_ctas) warm L2 before the programmatic-launch wait
  // Partial records per segment: C, or 1 when the C chunk CTAs of a segment form a
  // thread-block cluster and merge their partials through distributed shared memory.
  int32_t rps;
  float scale_log2;    // log2(e) / sqrt(d)
  int32_t B, Hq, Hkv, C;
  int32_t cu[FD_MAX_BATCH + 1];         // token prefix sums
  int32_t unit_base[FD_MAX_BATCH + 1];  // prefix sums of Hkv * W_b * C (CTA index base)
  uint16_t wseg[FD_MAX_BATCH];          // W_b
};
static_assert(sizeof(Params) <= 4096, "kernel parameters must stay within 4 KB");

// Token range of partial `slot` of a sequence of length L split into W segments
// of ceil(L/W) tokens, each cut into C chunks of ceil(n/C) tokens.  With align > 1
// (paged caches) both lengths are rounded up to multiples of `align` tokens.
FD_HD void chunk_range(int L, int W, int C, int slot, int align, int* t0, int* t1) {
  const int w = slot / C, c = slot - (slot / C) * C;
  int64_t S = L > 0 ? ((int64_t)L + W - 1) / W : 0;
  S = (S + align - 1) / align * align;
  int64_t sb = (int64_t)w * S;
  if (sb > L) sb = L;
  int64_t se = sb + S;
  if (se > L) se = L;
  const int64_t n = se - sb;
  const int64_t cl = ((n + C - 1) / C + align - 1) / align * align;
  int64_t a = (int64_t)c * cl, e = (int64_t)(c + 1) * cl;
  if (a > n) a = n;
  if (e > n) e = n;
  *t0 = (int)(sb + a);
  *t1 = (int)(sb + e);
}

// Launchers defined in the per-dtype kernel translation units.
// mode 0: fused split + last-arriver combine; 1: split only (partials); 2: combine only;
// 3: fused split + fine-grained waits (slot 0 combines partials as their flags arrive;
//    cooperative launch).
// pdl: launch with programmatic stream serialization (the kernel waits on its
// predecessors with griddepcontrol.wait before touching global memory).
cudaError_t launch_f16(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                       cudaStream_t s);
cudaError_t launch_bf16(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                        cudaStream_t s);

}  // namespace fd
