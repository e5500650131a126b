// Host side of the C ABI declared in include/fd.h: argument validation, the
// work decomposition (segments -> chunks -> CTAs), workspace layout, TMA
// tensor-map encoding and kernel launch.  See fd.h for the contract.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "fd_plan_internal.h"

namespace {

constexpr int kVersion = 0x000100;
constexpr size_t kAlign = 256;
// Auto chunking never cuts segments below this.  At 4K tokens with one query head per
// KV head (d = 64), 128-token chunks (256 CTAs) decode in 6.3 us against 7.7 us for
// 256-token chunks: the CUDA-core consumers of a CTA walk its tokens serially.
constexpr int kMinChunkTokens = 128;
constexpr int kMaxCluster = 8;        // portable thread-block cluster size
// CTAs that share one pair's combine unless the flags cap them: 8 for GQA groups of
// 8 or more (measured: the 128K-token G = 8 decode 79.4 against 80.0 us per step,
// 85.1 against 89.1 us alone; G = 16 at 32K 25.0 against 25.5 us, over an FP8 cache
// 18.9 against 20.9 us), the last arriver alone below (G = 4 at 32K: 22.7 against
// 22.6 us, 14.4 against 14.2 us over FP8).
constexpr int kDefaultCombiners = 8;
constexpr int kMinGroupForCombiners = 8;
// Plans whose CTAs read at most this many K/V bytes on average, and that have more
// CTAs than fit two per SM, run three CTAs per SM with 64 KB rings (fd_common.h).
constexpr int64_t kShallowMaxCtaBytes = 512 * 1024;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

// 3-D view (d, Hkv, N) of a [N, Hkv, d] tensor; one box = one tile of token rows of
// one head.  The MMA path loads 64-column boxes (128-byte rows) with the 128-byte
// swizzle; the FFMA path loads whole unswizzled rows.
int fd::encode_kv_map(CUtensorMap* map, const void* base, int64_t rows, int box_rows,
                      const fd_plan_s* pl) {
  auto enc = tensor_map_encoder();
  if (!enc) return FD_ERR_CUDA;
  const int es = fd::kv_elem_bytes(pl->path);
  const cuuint64_t dims[3] = {(cuuint64_t)pl->d, (cuuint64_t)pl->Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)pl->d * es, (cuuint64_t)pl->Hkv * pl->d * es};
  const cuuint32_t box[3] = {(cuuint32_t)fd::box_cols_for(pl->path, pl->d), 1u,
                             (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapDataType ty = pl->dtype == FD_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : pl->dtype == FD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle swz =
      fd::is_mma(pl->path) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = enc(map, ty, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FD_OK : FD_ERR_CUDA;
}

namespace {

cudaError_t launch(const fd_plan_s* pl, const fd::Params& p, int mode, int grid, cudaStream_t s) {
  return fd::launch_plan(pl, p, mode, grid, s);
}

}  // namespace

extern "C" {

int fd_version(void) { return kVersion; }

const char* fd_strerror(int status) {
  switch (status) {
    case FD_OK: return "FD_OK";
    case FD_ERR_INVALID: return "FD_ERR_INVALID: invalid argument";
    case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED: shape or option outside compiled support";
    case FD_ERR_ALIGN: return "FD_ERR_ALIGN: device pointer not 16-byte aligned";
    case FD_ERR_CUDA: return "FD_ERR_CUDA: CUDA call failed";
    case FD_ERR_NOMEM: return "FD_ERR_NOMEM: host allocation failed";
    case FD_ERR_STATE: return "FD_ERR_STATE: workspace counters not at rest";
    case FD_ERR_TIMEOUT: return "FD_ERR_TIMEOUT: bounded in-kernel wait gave up";
    default: return "unknown fd status";
  }
}

}  // extern "C"

namespace {

// fd_plan and fd_plan_paged: page_size == 0 plans the contiguous layout.
int plan_impl(int B, int Hq, int Hkv, int d, const int32_t* seqlens, const int32_t* W,
              int page_size, int dtype, uint32_t flags, int chunks, int num_sms,
              fd_plan_t* out_plan) {
  if (!out_plan) return FD_ERR_INVALID;
  *out_plan = nullptr;
  if (!seqlens || !W) return FD_ERR_INVALID;
  if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || chunks < 0 || num_sms < 0) return FD_ERR_INVALID;
  if (Hq % Hkv != 0) return FD_ERR_INVALID;
  if (dtype != FD_F16 && dtype != FD_BF16 && dtype != FD_F16_E4M3KV) return FD_ERR_INVALID;
  if (flags & ~(FD_PLAN_LITERAL_W | FD_PLAN_DEBUG | FD_PLAN_TWO_LAUNCH | FD_PLAN_FFMA |
                FD_PLAN_NO_PDL | FD_PLAN_WAITS | FD_PLAN_TEST_DROP_FLAG |
                FD_PLAN_NO_CLUSTER | FD_PLAN_CLUSTER | FD_PLAN_TEST_SKIP_TILE | FD_PLAN_TCGEN05 |
                FD_PLAN_CLUSTER_COMBINE | FD_PLAN_MMA_SYNC | FD_PLAN_COMBINERS_MASK |
                FD_PLAN_TEST_DROP_ARRIVAL | FD_PLAN_DEEP_RING))
    return FD_ERR_INVALID;
  const uint32_t combiners_code = (flags & FD_PLAN_COMBINERS_MASK) >> FD_PLAN_COMBINERS_SHIFT;
  if (combiners_code > 5) return FD_ERR_INVALID;
  if ((flags & FD_PLAN_CLUSTER) && (flags & (FD_PLAN_NO_CLUSTER | FD_PLAN_WAITS)))
    return FD_ERR_INVALID;
  if ((flags & FD_PLAN_WAITS) && (flags & FD_PLAN_TWO_LAUNCH)) return FD_ERR_INVALID;
  if ((flags & FD_PLAN_CLUSTER_COMBINE) &&
      (flags & (FD_PLAN_WAITS | FD_PLAN_TWO_LAUNCH | FD_PLAN_CLUSTER | FD_PLAN_NO_CLUSTER)))
    return FD_ERR_INVALID;
  if ((flags & FD_PLAN_TEST_DROP_FLAG) && !(flags & FD_PLAN_WAITS)) return FD_ERR_INVALID;
  if ((flags & FD_PLAN_TEST_DROP_FLAG) && (flags & FD_PLAN_TEST_SKIP_TILE)) return FD_ERR_INVALID;
  if ((flags & FD_PLAN_TEST_DROP_ARRIVAL) &&
      (flags & (FD_PLAN_WAITS | FD_PLAN_TWO_LAUNCH | FD_PLAN_CLUSTER_COMBINE | FD_PLAN_TEST_DROP_FLAG |
                FD_PLAN_TEST_SKIP_TILE)))
    return FD_ERR_INVALID;
  const int G = Hq / Hkv;
  if (page_size != 0 && (page_size < 16 || page_size > 256 || (page_size & (page_size - 1))))
    return FD_ERR_UNSUPPORTED;
  if (B > FD_MAX_BATCH) return FD_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FD_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return FD_ERR_UNSUPPORTED;
  if (G == 16 && (flags & FD_PLAN_FFMA)) return FD_ERR_UNSUPPORTED;  // tensor cores only
  if (dtype == FD_F16_E4M3KV && (d != 128 || G < 4 || (flags & FD_PLAN_FFMA)))
    return FD_ERR_UNSUPPORTED;
  if ((flags & FD_PLAN_TCGEN05) &&
      (dtype == FD_F16_E4M3KV || d != 128 || G < 4 || (flags & (FD_PLAN_FFMA | FD_PLAN_MMA_SYNC))))
    return FD_ERR_UNSUPPORTED;
  if ((flags & FD_PLAN_MMA_SYNC) && (flags & FD_PLAN_FFMA)) return FD_ERR_INVALID;
  // Tensor cores whenever the GQA group covers at least half of the mma N = 8 tile:
  // mma.sync by default, tcgen05 when asked for.  tcgen05 was the default for G = 16
  // until the combine was shared among the last arrivals: then two mma.sync N tiles
  // (256 CTAs, two per SM) decode 32K tokens in 24.2 us against 24.9 us on tcgen05
  // (128 CTAs, one per SM), the same box, three runs each.
  const bool umma = (flags & FD_PLAN_TCGEN05) != 0;
  const int path = dtype == FD_F16_E4M3KV                 ? fd::kPathMmaKv8
                   : umma                                 ? fd::kPathUmma
                   : (G >= 4 && !(flags & FD_PLAN_FFMA)) ? fd::kPathMma
                                                         : fd::kPathFfma;

  int64_t n_tokens = 0, sum_w = 0;
  int max_w = 0;
  for (int b = 0; b < B; ++b) {
    if (seqlens[b] < 0 || W[b] < 1) return FD_ERR_INVALID;
    if (W[b] > FD_MAX_PARTIALS) return FD_ERR_UNSUPPORTED;
    n_tokens += seqlens[b];
    sum_w += W[b];
    max_w = std::max(max_w, (int)W[b]);
  }
  if (n_tokens >= (int64_t)1 << 31) return FD_ERR_UNSUPPORTED;
  const bool pair = (flags & FD_PLAN_CLUSTER_COMBINE) != 0;
  if (pair) {
    // One cluster per (sequence, KV head): every sequence has the same W.
    for (int b = 1; b < B; ++b)
      if (W[b] != W[0]) return FD_ERR_UNSUPPORTED;
    if (W[0] > fd::kMaxPairCluster) return FD_ERR_UNSUPPORTED;
  }

  if (num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FD_ERR_CUDA;
    }
  }

  int C = 1;
  if (flags & FD_PLAN_LITERAL_W) {
    C = 1;
  } else if (chunks > 0) {
    C = chunks;
  } else {
    // Fill the resident CTA slots in one wave without cutting segments too short.
    const int64_t units = (int64_t)Hkv * sum_w;
    const int64_t slots = (int64_t)num_sms * fd::ctas_per_sm_for(path);
    int64_t c = std::max<int64_t>(1, slots / units);
    const int64_t avg_seg = sum_w > 0 ? n_tokens / sum_w : 0;
    c = std::min<int64_t>(c, std::max<int64_t>(1, avg_seg / kMinChunkTokens));
    if (pair) c = std::min<int64_t>(c, fd::kMaxPairCluster / W[0]);
    C = (int)c;
  }
  if (pair && (int64_t)W[0] * C > fd::kMaxPairCluster) return FD_ERR_UNSUPPORTED;
  if ((int64_t)max_w * C > FD_MAX_PARTIALS) return FD_ERR_UNSUPPORTED;
  {
    // The combine's shared-memory scratch must fit in the ring it reuses.
    const int64_t wt = (int64_t)max_w * C;
    int64_t need = (G * wt + 3 * G) * 4 + 16;                       // coefficients
    if (flags & FD_PLAN_WAITS)                                      // running state + lists
      need = std::max<int64_t>(need, (int64_t)(G * d + 4 * G + G * wt) * 4 + (2 * wt + 2) * 4);
    if (need > (int64_t)fd::ring_bytes_for(path, d, fd::ctas_per_sm_for(path))) return FD_ERR_UNSUPPORTED;
  }
  const int64_t ctas = (int64_t)Hkv * sum_w * C;
  if (ctas >= (int64_t)1 << 31) return FD_ERR_UNSUPPORTED;

  fd_plan_s* pl = new (std::nothrow) fd_plan_s();
  if (!pl) return FD_ERR_NOMEM;
  pl->B = B; pl->Hq = Hq; pl->Hkv = Hkv; pl->d = d; pl->G = G; pl->dtype = dtype;
  pl->flags = flags; pl->C = C; pl->num_sms = num_sms;
  pl->path = path;
  pl->page_size = page_size;
  pl->max_pages = 0;
  if (page_size)
    for (int b = 0; b < B; ++b)
      pl->max_pages = std::max(pl->max_pages, (seqlens[b] + page_size - 1) / page_size);
  pl->max_partials = max_w * C;
  pl->n_tokens = n_tokens;
  pl->total_partials = (int64_t)Hq * sum_w * C;
  pl->ctas = (int)ctas;

  fd::Params& p = pl->params;
  std::memset(&p, 0, sizeof(p));
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  p.test_hook = (flags & FD_PLAN_TEST_DROP_FLAG)      ? fd::kHookDropFlag
                : (flags & FD_PLAN_TEST_SKIP_TILE)    ? fd::kHookSkipTile
                : (flags & FD_PLAN_TEST_DROP_ARRIVAL) ? fd::kHookDropArrival
                                                      : fd::kHookNone;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.C = C;
  // The last arrivals of a pair share its combine by query heads only when every CTA
  // is resident at once (the CTAs they wait for then always run), in the fused
  // one-launch mode; never more combiners than partials.
  int nc = std::min(G, combiners_code            ? 1 << (combiners_code - 1)
                      : G >= kMinGroupForCombiners ? kDefaultCombiners
                                                   : 1);
  {
    const int64_t slots = (int64_t)num_sms * fd::ctas_per_sm_for(path);
    if ((flags & (FD_PLAN_TWO_LAUNCH | FD_PLAN_WAITS)) || pair || ctas > slots) nc = 1;
    while (nc > 1 && nc > max_w * C) nc >>= 1;
  }
  // When the chunk records one combiner reads would need several passes through the
  // combine's shared memory (at least 2; 3 over an FP8 cache, whose shorter CTAs
  // gain less than the cluster barriers cost), segments cut into 2..8 chunks merge
  // them inside a cluster (one record per segment); the last arriver then combines
  // alone.  Not in the fine-grained-waits variant, which combines chunk records as
  // they arrive.
  const int64_t rec_bytes = (int64_t)G / nc * max_w * C * fd::record_floats(d) * 4;
  const int64_t ring = (int64_t)fd::ring_bytes_for(pl->path, d, fd::ctas_per_sm_for(path));
  const bool multi_pass = rec_bytes > (pl->path == fd::kPathMmaKv8 ? 2 : 1) * ring;
  p.rps = ((multi_pass || (flags & FD_PLAN_CLUSTER)) && C > 1 && C <= kMaxCluster &&
           !(flags & (FD_PLAN_WAITS | FD_PLAN_NO_CLUSTER | FD_PLAN_CLUSTER_COMBINE))) ? 1 : C;
  if (p.rps != C) nc = 1;
  p.combiners = nc;
  // Many short CTAs on the fused mma.sync path, G <= 8 (more CTAs than two per SM,
  // at most kShallowMaxCtaBytes of K/V each): three CTAs per SM with 64 KB rings.
  {
    const int64_t kv_bytes = n_tokens * Hkv * d * 2 * fd::kv_elem_bytes(path);
    const int64_t slots = (int64_t)num_sms * fd::ctas_per_sm_for(path);
    const int64_t wt = (int64_t)max_w * C;
    const bool shallow =
        path == fd::kPathMma && G <= 8 && !pair && p.rps == C &&
        !(flags & (FD_PLAN_TWO_LAUNCH | FD_PLAN_WAITS | FD_PLAN_DEEP_RING)) && ctas > slots &&
        kv_bytes <= ctas * kShallowMaxCtaBytes &&
        (G * wt + 3 * G) * 4 + 16 <= (int64_t)fd::ring_bytes_for(path, d, fd::kShallowCtasPerSm);
    p.ctas_per_sm = shallow ? fd::kShallowCtasPerSm : fd::ctas_per_sm_for(path);
  }
  // Only the first wave can start before the previous kernel ends; later CTAs
  // would only queue prefetches ahead of their own loads.
  p.prefetch_ctas = (int32_t)std::min<int64_t>(ctas, (int64_t)num_sms * p.ctas_per_sm);
  p.pair_cluster = pair ? W[0] * C : 0;
  // Paged caches: boundaries on whole tiles, so that every TMA box stays in one page.
  p.align = page_size ? fd::tile_for(pl->path) : 1;
  p.box_rows = page_size ? std::min(fd::tile_for(pl->path), page_size) : fd::tile_for(pl->path);
  p.page_shift = 0;
  while (page_size && (1 << p.page_shift) < page_size) ++p.page_shift;
  int32_t cu = 0, ub = 0;
  for (int b = 0; b < B; ++b) {
    p.cu[b] = cu;
    p.unit_base[b] = ub;
    p.wseg[b] = (uint16_t)W[b];
    cu += seqlens[b];
    ub += Hkv * W[b] * C;
  }
  p.cu[B] = cu;
  p.unit_base[B] = ub;

  // Workspace: status | counters | flags | partial records [P][d + 4] (each 256-byte aligned).
  size_t off = kAlign;
  pl->off_counters = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)B * Hkv);
  pl->off_flags = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)pl->ctas);
  pl->off_part = off;
  off = align_up(off + sizeof(float) * (size_t)pl->total_partials * fd::record_floats(d));
  pl->ws_bytes = off;

  *out_plan = pl;
  return FD_OK;
}

}  // namespace

extern "C" {

int fd_plan(int B, int Hq, int Hkv, int d, const int32_t* seqlens, const int32_t* W, int dtype,
            uint32_t flags, int chunks, int num_sms, fd_plan_t* out_plan) {
  return plan_impl(B, Hq, Hkv, d, seqlens, W, 0, dtype, flags, chunks, num_sms, out_plan);
}

int fd_plan_paged(int B, int Hq, int Hkv, int d, const int32_t* seqlens, const int32_t* W,
                  int page_size, int dtype, uint32_t flags, int chunks, int num_sms,
                  fd_plan_t* out_plan) {
  if (page_size == 0) return FD_ERR_INVALID;
  return plan_impl(B, Hq, Hkv, d, seqlens, W, page_size, dtype, flags, chunks, num_sms,
                   out_plan);
}

int fd_plan_destroy(fd_plan_t plan) {
  delete plan;
  return FD_OK;
}

size_t fd_workspace_bytes(fd_plan_t plan) { return plan ? plan->ws_bytes : 0; }

int fd_plan_get_info(fd_plan_t pl, fd_plan_info* info) {
  if (!pl || !info) return FD_ERR_INVALID;
  info->B = pl->B; info->Hq = pl->Hq; info->Hkv = pl->Hkv; info->d = pl->d; info->G = pl->G;
  info->dtype = pl->dtype; info->flags = pl->flags; info->chunks = pl->C;
  info->num_sms = pl->num_sms; info->ctas = pl->ctas; info->max_partials = pl->max_partials;
  info->total_tokens = pl->n_tokens; info->total_partials = pl->total_partials;
  info->workspace_bytes = pl->ws_bytes;
  info->kv_bytes = (uint64_t)pl->n_tokens * pl->Hkv * pl->d * 2 * fd::kv_elem_bytes(pl->path);
  info->path = pl->path;
  info->records_per_segment = pl->params.rps;
  info->combine_cluster = pl->params.pair_cluster;
  info->combiners = pl->params.combiners;
  info->ctas_per_sm = pl->params.ctas_per_sm;
  return FD_OK;
}

int fd_plan_get_range(fd_plan_t pl, int b, int slot, int32_t* begin, int32_t* end) {
  if (!pl || !begin || !end || b < 0 || b >= pl->B) return FD_ERR_INVALID;
  const int wtot = pl->params.wseg[b] * pl->C;
  if (slot < 0 || slot >= wtot) return FD_ERR_INVALID;
  const int L = pl->params.cu[b + 1] - pl->params.cu[b];
  int t0, t1;
  fd::chunk_range(L, pl->params.wseg[b], pl->C, slot, pl->params.align, &t0, &t1);
  *begin = t0;
  *end = t1;
  return FD_OK;
}

int fd_workspace_init(fd_plan_t pl, void* workspace, cudaStream_t stream) {
  if (!pl || !workspace) return FD_ERR_INVALID;
  if (cudaMemsetAsync(workspace, 0, pl->off_part, stream) != cudaSuccess) {
    cudaGetLastError();
    return FD_ERR_CUDA;
  }
  return FD_OK;
}

int fd_workspace_status(fd_plan_t pl, void* workspace, cudaStream_t stream, int32_t* status) {
  if (!pl || !workspace || !status) return FD_ERR_INVALID;
  uint32_t word = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) {
    cudaGetLastError();
    return FD_ERR_CUDA;
  }
  *status = word == 0 ? FD_OK
          : (word & fd::kStatusTimeout) ? FD_ERR_TIMEOUT
                                        : FD_ERR_STATE;
  return FD_OK;
}

}  // extern "C"

namespace {

// fd_decode and fd_decode_paged.  `rows` is N (contiguous) or the page pool's
// num_pages * page_size rows; block_table is nullptr for the contiguous layout.
int decode_impl(fd_plan_t pl, const void* q, const void* k, const void* v, int64_t rows,
                const int32_t* block_table, int bt_stride, void* out, float* lse, void* workspace,
                cudaStream_t stream) {
  if (!pl || !q || !out || !workspace) return FD_ERR_INVALID;
  if (pl->n_tokens > 0 && (!k || !v)) return FD_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(workspace))
    return FD_ERR_ALIGN;

  fd::Params p = pl->params;  // per-call copy: the plan stays immutable
  if (pl->n_tokens > 0) {
    int rc = fd::encode_kv_map(&p.tm_k, k, rows, p.box_rows, pl);
    if (rc == FD_OK) rc = fd::encode_kv_map(&p.tm_v, v, rows, p.box_rows, pl);
    if (rc != FD_OK) return rc;
  }
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<uint32_t*>(ws + pl->off_counters);
  p.part = reinterpret_cast<float*>(ws + pl->off_part);
  p.flags = reinterpret_cast<uint32_t*>(ws + pl->off_flags);

  const bool debug = (pl->flags & FD_PLAN_DEBUG) != 0;
  if (debug) {
    std::vector<uint32_t> cnt((size_t)pl->B * pl->Hkv + 1);
    if (cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaMemcpy(cnt.data(), p.counters, sizeof(uint32_t) * (cnt.size() - 1),
                   cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return FD_ERR_CUDA;
    }
    for (size_t i = 0; i + 1 < cnt.size(); ++i)
      if (cnt[i] != 0) return FD_ERR_STATE;
  }

  cudaError_t err;
  if (pl->flags & FD_PLAN_TWO_LAUNCH) {
    err = launch(pl, p, 1, pl->ctas, stream);
    if (err == cudaSuccess) err = launch(pl, p, 2, pl->B * pl->Hkv, stream);
  } else {
    err = launch(pl, p, fd::fused_mode(pl), pl->ctas, stream);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fd::launch_status(err);
  }
  if (debug) {
    int32_t st = FD_OK;
    int rc = fd_workspace_status(pl, workspace, stream, &st);
    if (rc != FD_OK) return rc;
    if (st != FD_OK) return st;
  }
  return FD_OK;
}

}  // namespace

extern "C" {

int fd_decode(fd_plan_t pl, const void* q, const void* k, const void* v, void* out, float* lse,
              void* workspace, cudaStream_t stream) {
  if (pl && pl->page_size != 0) return FD_ERR_INVALID;  // paged plans use fd_decode_paged
  return decode_impl(pl, q, k, v, pl ? pl->n_tokens : 0, nullptr, 0, out, lse, workspace, stream);
}

int fd_decode_paged(fd_plan_t pl, const void* q, const void* k_pages, const void* v_pages,
                    int num_pages, const int32_t* block_table, int bt_stride, void* out, float* lse,
                    void* workspace, cudaStream_t stream) {
  if (!pl || pl->page_size == 0) return FD_ERR_INVALID;
  if (pl->n_tokens > 0) {
    if (num_pages < 1 || !block_table || bt_stride < pl->max_pages) return FD_ERR_INVALID;
    if ((int64_t)num_pages * pl->page_size >= (int64_t)1 << 31) return FD_ERR_UNSUPPORTED;
  }
  return decode_impl(pl, q, k_pages, v_pages, (int64_t)num_pages * pl->page_size, block_table,
                     bt_stride, out, lse, workspace, stream);
}

}  // extern "C"
