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
// UMMA: fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory),
// d = 128 and G in {4, 8, 16}: S^T = K Q^T with 128 tokens on M and the heads
// (padded to 16) on N, read straight from the TMA-swizzled K tile; P^T goes through
// shared memory; O^T = V^T P^T accumulates in tensor memory with the 128 head
// dimensions on M.  K and V tiles of 128 tokens occupy separate ring slots.
constexpr int kPathFfma = 0;
constexpr int kPathMma = 1;
constexpr int kPathMmaKv8 = 2;
constexpr int kPathUmma = 3;

FD_HD constexpr bool is_mma(int path) { return path != kPathFfma; }
// Bytes per stored K/V element.
FD_HD constexpr int kv_elem_bytes(int path) { return path == kPathMmaKv8 ? 1 : 2; }
// Tokens per pipeline stage.
// (FP8: 128-token tiles, two 16-token groups per consumer warp per stage.)
FD_HD constexpr int tile_for(int path) {
  return (path == kPathUmma || path == kPathMmaKv8) ? 128 : is_mma(path) ? 64 : 32;
}
// Columns (elements) of one TMA box row: 128-byte swizzled rows on the MMA paths.
FD_HD constexpr int box_cols_for(int path, int d) {
  return (path == kPathMma || path == kPathUmma) ? 64 : path == kPathMmaKv8 ? 128 : d;
}
// Ring slots per tile: the tcgen05 path keeps K and V of a tile in separate slots
// (the K slot is released when S^T is computed, the V slot after P.V).
FD_HD constexpr int loads_per_tile(int path) { return path == kPathUmma ? 2 : 1; }
// K/V tokens per CTA that the split kernel prefetches into L2 before it waits for
// the previous kernel in the stream (256 = 4 tiles of 64 measured best for fp16 and
// fp8 caches at 32K and 128K tokens; 2 and 8 tiles were slower).
constexpr int kL2PrefetchTokens = 256;
// The K/V ring, 96 KB on every path: slots of one tile of K rows followed by the
// tile of V rows of one KV head.  (At d = 64 the ring used to be 64 KB; 96 KB is
// 14% faster at 32K tokens.  A 112 KB ring, the most two CTAs per SM can hold,
// was slower on every path, and so were separate K and V slots with their own
// barriers on the multi-wave and FP8 cases.)
constexpr int kRingBytes = 96 * 1024;
// A kernel that uses tcgen05 instructions is resident one CTA per SM (the occupancy
// calculator reports 1 for any such kernel, whatever its shared memory), so that
// path gets the bytes in flight of two CTAs of the other paths: a 192 KB ring.
FD_HD constexpr int ctas_per_sm_for(int path) { return path == kPathUmma ? 1 : 2; }
// Plans of many short CTAs on the mma.sync path run three CTAs per SM with 64 KB
// rings instead (kShallowCtasPerSm): one CTA's ramp and tail then leave two others
// streaming.  (Measured on 64 sequences of 8K tokens: 512-token CTAs 305.2 against
// 314.2 us, 1024-token CTAs 299.8 against 301.2 us; 2048 tokens even; 4096 and more
// tokens per CTA, and every one-wave plan, slower.)
constexpr int kShallowCtasPerSm = 3;
constexpr int kShallowRingBytes = 64 * 1024;
FD_HD constexpr int ring_target_bytes(int path, int cps) {
  return path == kPathUmma ? 2 * kRingBytes : cps == kShallowCtasPerSm ? kShallowRingBytes : kRingBytes;
}
FD_HD constexpr int slot_bytes_for(int path, int d) {
  return (2 / loads_per_tile(path)) * tile_for(path) * d * kv_elem_bytes(path);
}
// `cps`: resident CTAs per SM the kernel is built for (ctas_per_sm_for, or
// kShallowCtasPerSm).
FD_HD constexpr int ring_slots_for(int path, int d, int cps) {
  return ring_target_bytes(path, cps) / slot_bytes_for(path, d);
}
// Bytes of the K/V ring (also the scratch the combine reuses).
FD_HD constexpr size_t ring_bytes_for(int path, int d, int cps) {
  return (size_t)ring_slots_for(path, d, cps) * slot_bytes_for(path, d);
}
// Bytes after the ring: 2 mbarriers per slot, an unused word, two flags, the
// tcgen05 path's two mbarriers and tensor-memory address, the combine's 16
// mbarriers (one per head of a pass), and up to 1 KB of slack for aligning the ring
// to 1024 bytes.
constexpr int kRingMetaBytes = 2048;
// The tcgen05 path's operands outside the ring: Q (16 x 128, 4 KB), P^T (128 x 16,
// 4 KB), 1 KB of reduction scratch, and P^T's low part for bf16 weights (4 KB).
FD_HD constexpr int extra_bytes_for(int path) { return path == kPathUmma ? 13312 : 0; }
// Dynamic shared memory of one CTA: the ring, the extra operands and the metadata.
FD_HD constexpr size_t smem_bytes_for(int path, int d, int cps) {
  return ring_bytes_for(path, d, cps) + extra_bytes_for(path) + kRingMetaBytes;
}
// Floats per partial record: O[0..d), m, l, l~ and a pad word (16-byte records).
// l sums the fp32 softmax weights (it gives lse); l~ sums the weights as rounded
// for the P.V product (it normalises out, so out is an exact convex combination
// of V rows under those weights).  Without rounding (CUDA-core path) l~ = l.
FD_HD constexpr int record_floats(int d) { return d + 4; }

// Largest cluster of the pair-cluster combine (FD_PLAN_CLUSTER_COMBINE): the
// non-portable cluster size limit.
constexpr int kMaxPairCluster = 16;

// Status word values written by the kernels (the host maps them to fd_status).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusCounter = 2u;

// Test hooks (chosen by plan flags) that make one bounded wait run out on purpose.
// kHookDropFlag: partial slot 1 of (sequence 0, KV head 0) never sets its ready flag
// (fine-grained-waits variant).  kHookSkipTile: the producer of partial slot 0 of
// (sequence 0, KV head 0) never issues the loads of its second tile, so that CTA's
// consumers give up waiting for it.  kHookDropArrival: partial slot 1 of (sequence 0,
// KV head 0) never arrives, so the pair's combiners give up waiting for the last one.
constexpr int32_t kHookNone = 0;
constexpr int32_t kHookDropFlag = 1;
constexpr int32_t kHookSkipTile = 2;
constexpr int32_t kHookDropArrival = 3;

// Kernel parameters (passed by value as a __grid_constant__ struct; < 4 KB).
struct Params {
  CUtensorMap tm_k;  // 3-D view of K: (d, Hkv, N), box (d, 1, kTile)
  CUtensorMap tm_v;  // same for V
  const void* q;     // [B, Hq, d]
  void* out;         // [B, Hq, d]
  float* lse;        // [B, Hq] or nullptr
  float* part;       // [P, d + 4] records: O[0..d), m, l, l~, 0 (m in the log2 domain)
  uint32_t* counters;  // [B * Hkv]
  uint32_t* flags;     // [CTAs] per-partial ready flags (fine-grained-waits variant)
  uint32_t* status;    // 1 word
  int32_t test_hook;   // kHookNone, or one of the test hooks below
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
  // CTAs per cluster when every partial of a (sequence, KV head) pair forms one
  // cluster and combines there (kernel mode 6): W * C, equal for every sequence.
  int32_t pair_cluster;
  // CTAs that share the combine of one (sequence, KV head) pair: the last
  // `combiners` arrivals (a power of two dividing G; 1 = the last arriver alone).
  int32_t combiners;
  // Resident CTAs per SM the split kernel is launched for: ctas_per_sm_for(path), or
  // kShallowCtasPerSm (64 KB rings) for plans of many short CTAs on the mma.sync path.
  int32_t ctas_per_sm;
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

// Launchers defined in the kernel translation units (one per dtype and consumer family).
// mode 0: fused split + last-arriver combine; 1: split only (partials); 2: combine only;
// 3: fused split + fine-grained waits (slot 0 combines partials as their flags arrive;
//    cooperative launch); 6: fused, every partial of a (sequence, KV head) pair in one
//    thread-block cluster, combined through distributed shared memory.
// pdl: launch with programmatic stream serialization (the kernel waits on its
// predecessors with griddepcontrol.wait before touching global memory).
cudaError_t launch_f16_mma(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                           cudaStream_t s);
cudaError_t launch_bf16_mma(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                            cudaStream_t s);
cudaError_t launch_f16_ffma(const Params& p, int d, int G, int mode, bool pdl, int grid,
                            cudaStream_t s);
cudaError_t launch_bf16_ffma(const Params& p, int d, int G, int mode, bool pdl, int grid,
                             cudaStream_t s);
cudaError_t launch_umma_f16(const Params& p, int d, int G, int mode, bool pdl, int grid,
                            cudaStream_t s);
cudaError_t launch_umma_bf16(const Params& p, int d, int G, int mode, bool pdl, int grid,
                             cudaStream_t s);

}  // namespace fd
