/*
 * fd.h -- C ABI of the GB300 split-KV Flash Decode library (libfd_gb300.so).
 *
 * The operation ("Eliminating Multi-GPU Performance Taxes", review page:
 * notation table and core equations, "Flash Decode global reduction"):
 * one query token per sequence attends over that sequence's KV cache, which
 * is split into W segments; each segment yields a partial (O, m, l) and the
 * partials are merged by OnlineSoftmaxCombine, whose associativity lets them
 * be merged in any order (correctness check #5, Milakov & Gimelshein 2018).
 * Here the W segments are splits of one GPU's KV cache.  fd_decode runs the
 * whole path in ONE kernel launch: every CTA streams its K/V rows through a
 * TMA/mbarrier shared-memory ring, computes its partial, publishes it, and the
 * CTA that arrives last for a (sequence, KV head) combines all partials of
 * that pair (the pages' "fully fused" variant, with a release/acquire arrival
 * counter in place of the pages' remote inbox flags).  When the whole grid is
 * resident at once, the last few CTAs to arrive share that combine, each taking
 * a slice of the pair's query heads (fd_plan_info.combiners).
 *
 * Result, for sequence b, query head h, KV head g = h / (Hq / Hkv):
 *   s_j = <q[b,h,:], K[cu_b + j, g, :]> / sqrt(d),  j = 0 .. L_b - 1
 *   out[b,h,:] = sum_j softmax(s)_j V[cu_b + j, g, :]     (stored in q's type)
 *   lse[b,h]   = ln sum_j exp(s_j)                        (fp32, natural log)
 * with fp32 accumulation.  L_b = 0 gives out = 0 and lse = -inf.
 *
 * Conventions for every entry point:
 *   - Every call returns an int status (enum fd_status).  Nothing aborts and
 *     nothing throws across the ABI.  fd_strerror() names a status.
 *   - Device pointers belong to the calling thread's current CUDA device.
 *   - Calls that take a stream are asynchronous with respect to the host unless
 *     stated otherwise; a launch error is reported as FD_ERR_CUDA.
 */
#ifndef FD_GB300_FD_H_
#define FD_GB300_FD_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque, immutable plan.  Owns host memory only.  A plan may be shared by
 * threads; one workspace serves one in-flight decode at a time. */
typedef struct fd_plan_s* fd_plan_t;

enum fd_dtype {
  FD_F16 = 0,        /* IEEE binary16 q, K, V and out */
  FD_BF16 = 1,       /* bfloat16 q, K, V and out */
  /* binary16 q and out over an FP8 cache: K and V are OCP FP8 E4M3 bytes (no
   * per-tensor scale: a scaled cache folds its K scale into q and its V scale
   * into out).  Needs d = 128 and G >= 4 (tensor-core path); the K/V bytes per
   * token halve. */
  FD_F16_E4M3KV = 2
};

enum fd_status {
  FD_OK = 0,
  FD_ERR_INVALID = -1,     /* bad argument (null pointer, negative size, Hq % Hkv != 0, ...) */
  FD_ERR_UNSUPPORTED = -2, /* valid but outside the compiled support (d, G, batch, partial count) */
  FD_ERR_ALIGN = -3,       /* a device pointer is not 16-byte aligned */
  FD_ERR_CUDA = -4,        /* a CUDA runtime or driver call failed */
  FD_ERR_NOMEM = -5,       /* host allocation failed */
  FD_ERR_STATE = -6,       /* workspace counters not at rest (debug plans check this) */
  FD_ERR_TIMEOUT = -7      /* a bounded in-kernel wait gave up (device status word) */
};

/* fd_plan flags */
#define FD_PLAN_LITERAL_W 0x1u /* exactly W_b partials per sequence (chunks = 1) */
#define FD_PLAN_DEBUG 0x2u     /* fd_decode checks counters/status (synchronises the stream) */
#define FD_PLAN_TWO_LAUNCH 0x4u /* split kernel + separate combine kernel (ablation) */
#define FD_PLAN_FFMA 0x8u       /* CUDA-core scores and P.V even when G >= 4 (ablation) */
#define FD_PLAN_NO_PDL 0x10u    /* launch without programmatic dependent launch (ablation) */
/* Fine-grained waits (the pages' V3 reading): partial slot 0 of every (sequence,
 * KV head) waits on per-partial ready flags and combines partials as they arrive.
 * Cooperative launch: FD_ERR_UNSUPPORTED when the grid cannot be co-resident.
 * The combine order follows arrival, so results are not bitwise reproducible. */
#define FD_PLAN_WAITS 0x20u
/* Test hook for FD_PLAN_WAITS: partial slot 1 of (sequence 0, KV head 0) never
 * sets its flag, so that combiner's bounded wait runs out (~1 s) and the status
 * word reports FD_ERR_TIMEOUT.  Its out/lse are left unwritten. */
#define FD_PLAN_TEST_DROP_FLAG 0x40u
/* Segment merge.  When the planner cuts each segment into 2..8 chunks, the chunk
 * CTAs of a segment can run as one thread-block cluster and merge their partials
 * through distributed shared memory, so that the combine reads one record per
 * segment, as in the pages.  By default this happens when one (sequence, KV head)'s
 * chunk records would not fit the combine's shared memory in one pass.
 * FD_PLAN_NO_CLUSTER never merges; FD_PLAN_CLUSTER always does (both: invalid). */
#define FD_PLAN_NO_CLUSTER 0x80u
#define FD_PLAN_CLUSTER 0x100u
/* Test hook for the pipeline's bounded waits: the producer of partial slot 0 of
 * (sequence 0, KV head 0) never loads that partial's second tile, so its
 * consumers give up after ~1 s.  That CTA then publishes an empty partial and
 * still arrives, so every arrival counter returns to zero; the status word
 * reports FD_ERR_TIMEOUT and the out/lse of (sequence 0, KV head 0) lack that
 * partial.  Needs L_0 large enough for slot 0 to span two tiles (128 tokens with
 * FD_PLAN_TCGEN05 or an E4M3 cache, 64 on the other tensor-core paths, 32 on CUDA
 * cores); otherwise nothing is skipped.  Not with FD_PLAN_TEST_DROP_FLAG. */
#define FD_PLAN_TEST_SKIP_TILE 0x200u
/* Test hook for the shared combine's bounded wait: partial slot 1 of (sequence 0, KV
 * head 0) publishes its partial but never arrives.  The combiners of that pair wait
 * for the last arrival, give up after ~4 s and report FD_ERR_TIMEOUT in the status
 * word; the pair's out/lse are not written, and its counter is left short, so the
 * workspace needs fd_workspace_init before the next decode.  Only meaningful for a
 * plan with fd_plan_info.combiners > 1 (with a single combiner nothing waits and the
 * pair is simply never combined).  Not with FD_PLAN_WAITS, FD_PLAN_TWO_LAUNCH,
 * FD_PLAN_CLUSTER_COMBINE or the other test hooks. */
#define FD_PLAN_TEST_DROP_ARRIVAL 0x2000u
/* Keep two CTAs per SM with 96 KB K/V rings (ablation).  Without it, a plan on the
 * mma.sync path (G = 4 or 8, 16-bit K/V) whose CTAs do not all fit two per SM and read
 * at most 512 KB of K/V each on average, run as one fused launch without clusters,
 * runs three CTAs per SM with 64 KB rings: one CTA's ramp and tail then leave two
 * others streaming (fd_plan_info.ctas_per_sm). */
#define FD_PLAN_DEEP_RING 0x4000u
/* Fifth-generation tensor cores (tcgen05.mma with accumulators in tensor memory)
 * for the scores and P.V: 128-token tiles, d = 128, G in {4, 8, 16}, fp16 or bf16
 * (FD_ERR_UNSUPPORTED otherwise).  Not the default: mma.sync measured faster on
 * every decode case measured once the combine is shared (G = 16 at 32K tokens: 24.9
 * against 24.2 us).  A kernel with tcgen05 instructions is resident one CTA per SM, so these
 * plans size their grid for one CTA per SM and give it a 192 KB K/V ring.
 * S^T = K Q^T runs with the tokens on M and the heads, padded to 16, on N, straight
 * from the TMA-swizzled K tile; P^T is staged in shared memory; O^T = V^T P^T
 * accumulates in tensor memory. */
#define FD_PLAN_TCGEN05 0x400u
/* Combine in a thread-block cluster: the W * C partial CTAs of each (sequence, KV
 * head) pair run as one cluster (at most 16 CTAs), keep their partials in shared
 * memory and, after a cluster barrier, each combines its share of the pair's output
 * columns from all partials through distributed shared memory.  No partial record,
 * counter or flag touches global memory.  Needs the same W for every sequence and
 * W <= 16 (FD_ERR_UNSUPPORTED otherwise); the planner caps C at 16 / W.  Not with
 * FD_PLAN_WAITS, FD_PLAN_TWO_LAUNCH, FD_PLAN_CLUSTER or FD_PLAN_NO_CLUSTER.  A
 * device that cannot place the clusters makes fd_decode return FD_ERR_UNSUPPORTED. */
#define FD_PLAN_CLUSTER_COMBINE 0x800u
/* The mma.sync tensor-core consumers (the default for G >= 4; the flag pins that
 * choice).  Not with FD_PLAN_TCGEN05 or FD_PLAN_FFMA. */
#define FD_PLAN_MMA_SYNC 0x1000u
/* Cap on the CTAs that share the combine of one (sequence, KV head) pair, in bits
 * 16..18 of the flags: FD_PLAN_COMBINERS_n allows at most n.  Without one, the
 * planner allows 8 for G >= 8 and 1 below.  A plan whose CTAs all fit on the
 * device at once (at most SMs x resident CTAs per SM), run as one fused launch
 * without clusters, lets the last `combiners` arrivals of each pair share its
 * combine: the r-th CTA before the last waits (bounded, ~4 s) until the last one
 * has arrived, then combines query heads [r * G / combiners, (r + 1) * G /
 * combiners).  Each head is combined by the same code either way, so the results
 * are bit-identical.  FD_PLAN_SINGLE_COMBINER (the last arriver alone) is the
 * ablation.  num_sms must not exceed the device's SM count for such plans: a
 * combiner could otherwise wait for a CTA that has no SM to run on, until its
 * bounded wait gives up (FD_ERR_TIMEOUT). */
#define FD_PLAN_COMBINERS_SHIFT 16
#define FD_PLAN_COMBINERS_MASK (7u << FD_PLAN_COMBINERS_SHIFT)
#define FD_PLAN_COMBINERS_1 (1u << FD_PLAN_COMBINERS_SHIFT)
#define FD_PLAN_COMBINERS_2 (2u << FD_PLAN_COMBINERS_SHIFT)
#define FD_PLAN_COMBINERS_4 (3u << FD_PLAN_COMBINERS_SHIFT)
#define FD_PLAN_COMBINERS_8 (4u << FD_PLAN_COMBINERS_SHIFT)
#define FD_PLAN_COMBINERS_16 (5u << FD_PLAN_COMBINERS_SHIFT)
#define FD_PLAN_SINGLE_COMBINER FD_PLAN_COMBINERS_1

/* Compiled limits. */
#define FD_MAX_BATCH 256       /* sequences per plan */
#define FD_MAX_PARTIALS 1024   /* W_b * chunks per sequence */

/*
 * fd_plan -- validate a decode shape and build its work decomposition (host only;
 * no CUDA call unless num_sms == 0).
 *
 *   B        number of sequences, 1 .. FD_MAX_BATCH
 *   Hq, Hkv  query / KV heads; Hq % Hkv == 0; G = Hq / Hkv in {1, 2, 4, 8, 16}
 *            (G >= 4 runs on tensor cores; G = 16 only there)
 *   d        head dimension, 64 or 128
 *   seqlens  host array [B], L_b >= 0; sum_b L_b < 2^31.  Sequence b occupies
 *            KV rows [cu_b, cu_b + L_b) with cu_b = L_0 + ... + L_{b-1}.
 *   W        host array [B], W_b >= 1 segments for sequence b.  Segment w is
 *            [w*S_b, min((w+1)*S_b, L_b)) with S_b = ceil(L_b / W_b); trailing
 *            segments may be empty (the pages shard the KV cache W ways; this
 *            split rule is the plan's reading).
 *   dtype    enum fd_dtype (q / out type; K / V the same, or E4M3 bytes)
 *   flags    FD_PLAN_* bits
 *   chunks   chunks per segment C >= 1 (each segment is cut into C equal
 *            pieces, so W_b * C partials are combined); 0 = choose from the
 *            SM count.  Ignored (C = 1) with FD_PLAN_LITERAL_W.
 *   num_sms  SM count used to choose C; 0 = query the current device
 *            (FD_ERR_CUDA if there is none).
 *   out_plan receives the plan; release it with fd_plan_destroy.
 *
 * The plan copies seqlens and W; the caller keeps ownership of its arrays.
 */
int fd_plan(int B, int Hq, int Hkv, int d, const int32_t* seqlens, const int32_t* W,
            int dtype, uint32_t flags, int chunks, int num_sms, fd_plan_t* out_plan);

/*
 * fd_plan_paged -- fd_plan for a paged KV cache (block tables; a deployment
 * layout the pages do not discuss).  Same arguments plus
 *   page_size  tokens per page: a power of two in [16, 256]
 * Segment and chunk lengths are rounded up to whole kernel tiles (64 tokens on
 * the tensor-core path, 32 on CUDA cores) so that every TMA box stays inside one
 * page; the split changes, the result does not (the combine is exact for any
 * partition).  Decode with fd_decode_paged.
 */
int fd_plan_paged(int B, int Hq, int Hkv, int d, const int32_t* seqlens, const int32_t* W,
                  int page_size, int dtype, uint32_t flags, int chunks, int num_sms,
                  fd_plan_t* out_plan);

/* Release a plan (NULL is accepted).  No CUDA call. */
int fd_plan_destroy(fd_plan_t plan);

/* Bytes of device workspace fd_decode needs for this plan: a status word, one
 * uint32 arrival counter per (sequence, KV head), one uint32 ready flag per CTA,
 * and the fp32 partial records [P][d + 4] (O, m, l, l~; P = Hq * sum_b W_b * C).
 * 0 for a NULL plan. */
size_t fd_workspace_bytes(fd_plan_t plan);

/* Zero the workspace's counters, flags and status word on `stream` (asynchronous).
 * A workspace must be zeroed once before its first fd_decode (torch.zeros or
 * this call); fd_decode leaves every counter at zero when it completes. */
int fd_workspace_init(fd_plan_t plan, void* workspace, cudaStream_t stream);

/*
 * fd_decode -- the fused split-KV Flash Decode (one kernel launch on `stream`).
 *
 *   q          device [B, Hq, d] (dtype), contiguous
 *   k, v       device [N, Hkv, d] (dtype; 1-byte E4M3 for FD_F16_E4M3KV), contiguous,
 *              N = sum_b L_b
 *   out        device [B, Hq, d] (dtype), written
 *   lse        device [B, Hq] float, written (natural log); may be NULL
 *   workspace  device, fd_workspace_bytes(plan) bytes, zeroed once beforehand
 *   stream     CUDA stream (0 = legacy default stream)
 *
 * All device pointers must be 16-byte aligned (FD_ERR_ALIGN otherwise).  The
 * caller owns every buffer and the stream.  Kernels are launched with
 * programmatic dependent launch (unless FD_PLAN_NO_PDL): their prologue may
 * overlap the previous kernel on the stream, but they read and write global
 * memory only after every earlier kernel has completed.  The prologue does
 * prefetch the first K/V tiles of each chunk into L2 (contiguous layout only); a
 * prefetch returns no data, so it cannot observe a K/V write still in flight.  Asynchronous: returns after the
 * launch; with FD_PLAN_DEBUG it synchronises and reports FD_ERR_TIMEOUT or
 * FD_ERR_STATE from the device status word.  Decodes that share a workspace
 * must not overlap in time.
 */
int fd_decode(fd_plan_t plan, const void* q, const void* k, const void* v, void* out,
              float* lse, void* workspace, cudaStream_t stream);

/*
 * fd_decode_paged -- fd_decode over a paged KV cache.
 *
 *   k_pages, v_pages  device [num_pages, page_size, Hkv, d] (dtype), contiguous pools
 *   num_pages         pages in each pool (num_pages * page_size < 2^31)
 *   block_table       device int32 [B, bt_stride]: row b lists, in order, the pool
 *                     pages holding tokens [j*page_size, (j+1)*page_size) of
 *                     sequence b, for j < ceil(L_b / page_size)
 *   bt_stride         entries per row, >= max_b ceil(L_b / page_size)
 *   q, out, lse, workspace, stream   as for fd_decode
 *
 * Returns FD_ERR_INVALID for a contiguous plan or a short bt_stride.  Page
 * indices outside [0, num_pages) read zeros (TMA out-of-bounds fill); they never
 * fault, but the result is then meaningless.  fd_decode rejects paged plans.
 */
int fd_decode_paged(fd_plan_t plan, const void* q, const void* k_pages, const void* v_pages,
                    int num_pages, const int32_t* block_table, int bt_stride, void* out,
                    float* lse, void* workspace, cudaStream_t stream);

/* Bytes of the static device scratch array behind fd_decode_noalloc (32 MiB). */
#define FD_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * fd_decode_noalloc -- fd_decode for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for deployment.
 *
 * Who needs it: code that runs inside an engine or framework owning the device
 * allocator (a plugin enqueue that must not call cudaMalloc, a caching-allocator
 * arena that must not fragment), or any call site where a device allocation
 * would synchronise the device.  Such callers cannot provide fd_decode's
 * workspace.  This call takes none: the counters, status word and fp32
 * partials live in one file-scope __device__ array of FD_NOALLOC_SCRATCH_BYTES
 * that every GPU loading the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine);
 * the plan comes from fd_plan, which allocates host memory only.
 *
 *   plan, q, k, v, out, lse, stream   as for fd_decode (no workspace argument)
 *
 * Returns FD_ERR_UNSUPPORTED when fd_workspace_bytes(plan) exceeds
 * FD_NOALLOC_SCRATCH_BYTES (the plan needs more scratch than the array holds).
 * The device address of the array is looked up (cudaGetSymbolAddress, with that
 * device current) by the first call in each CUDA context of a device, and again
 * after the context changes (e.g. after cudaDeviceReset); make that first call
 * before any stream capture.  Each call clears the array's status word,
 * counters and flags on `stream` before its launch; the array keeps the last
 * call's partials.  Every call in the process shares the one array per device,
 * so fd_decode_noalloc calls that overlap on the GPU (other streams, other
 * threads) race and must be serialised by the caller.  A bounded in-kernel wait
 * that gives up is reported by fd_noalloc_status (read it before the next call,
 * which clears it); with FD_PLAN_DEBUG this call synchronises and returns that
 * status itself.  Asynchronous otherwise, like fd_decode.
 */
int fd_decode_noalloc(fd_plan_t plan, const void* q, const void* k, const void* v, void* out,
                      float* lse, cudaStream_t stream);

/*
 * fd_noalloc_status -- the device status of the last fd_decode_noalloc call on the
 * current device (the paper has no counterpart; it serves fd_decode_noalloc).
 * Synchronises `stream`, reads the static array's status word and the plan's
 * counters and ready flags, then clears the status word.  *status is FD_OK,
 * FD_ERR_TIMEOUT (a bounded wait gave up) or FD_ERR_STATE (a counter overflowed,
 * or counters or flags are not back at zero).  Allocates nothing.
 * FD_ERR_UNSUPPORTED for a plan whose scratch exceeds the array.
 */
int fd_noalloc_status(fd_plan_t plan, cudaStream_t stream, int32_t* status);

/* Synchronise `stream` and read the device status word (0 = no error; else a
 * negative fd_status) into *status.  Then clear the word. */
int fd_workspace_status(fd_plan_t plan, void* workspace, cudaStream_t stream,
                        int32_t* status);

/* Human-readable name of a status code (static string, never NULL). */
const char* fd_strerror(int status);

/* Plan introspection (host only). */
typedef struct fd_plan_info {
  int32_t B, Hq, Hkv, d, G, dtype;
  uint32_t flags;
  int32_t chunks;          /* C actually used */
  int32_t num_sms;         /* SM count the plan was sized for */
  int32_t ctas;            /* CTAs fd_decode launches = Hkv * sum_b W_b * C */
  int32_t max_partials;    /* max_b W_b * C */
  int64_t total_tokens;    /* N */
  int64_t total_partials;  /* P */
  uint64_t workspace_bytes;
  uint64_t kv_bytes;       /* bytes of K and V one decode reads */
  int32_t path;            /* 0: CUDA-core (FFMA) consumers, 1: tensor-core (mma.sync),
                              2: tensor-core over an E4M3 cache, 3: tcgen05 tensor cores */
  int32_t records_per_segment; /* partial records per segment: 1 (chunks merged in a
                                  cluster) or chunks */
  int32_t combine_cluster; /* CTAs per cluster that combine a pair's partials in shared
                              memory (FD_PLAN_CLUSTER_COMBINE: W * chunks), else 0 */
  int32_t combiners;       /* CTAs that share the combine of one pair: a power of two
                              dividing G (fewer for a sequence with fewer partials),
                              1 = the last arriver alone */
  int32_t ctas_per_sm;     /* resident CTAs per SM the split kernel is launched for:
                              2 (96 KB rings), 3 (64 KB rings) or 1 (tcgen05) */
} fd_plan_info;

int fd_plan_get_info(fd_plan_t plan, fd_plan_info* info);

/* Token range [*begin, *end) (relative to the start of sequence b) covered by
 * partial `slot` (0 <= slot < W_b * C) of sequence b. */
int fd_plan_get_range(fd_plan_t plan, int b, int slot, int32_t* begin, int32_t* end);

/* Library version, e.g. 0x000100 for 0.1.0. */
int fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_GB300_FD_H_ */
