// Fused split-KV Flash Decode for sm_103a.
//
// Method ("Eliminating Multi-GPU Performance Taxes", review page): single-token
// attention whose KV cache is split into W segments; every segment produces a
// partial (O, m, l) and OnlineSoftmaxCombine merges the partials, in any order
// (core equations, "Flash Decode global reduction"; correctness check #5).  The
// pages' fastest variant ("Fully Fused Kernels", ablation table) fuses the
// partial computation and the reduction into one kernel in which producers
// publish data, then a flag, and consumers combine what has arrived
// (Push-model flag ordering, correctness check #4).
//
// GB300 mapping (one CTA = one chunk of one segment of one (sequence, KV head)):
//   * warp 4, lane 0: TMA producer.  Before the programmatic-launch wait, CTAs
//     of the first wave prefetch the first tiles of their chunk into L2 (HBM is
//     idle while the previous decode combines).  Per stage it issues 3-D tensor
//     loads of a tile of K rows and of V rows of one KV head into an mbarrier ring.
//   * warps 0-3: consumers; every K/V byte loaded serves all G query heads that
//     share the KV head (GQA packing).  Two consumer paths:
//       MMA  (G >= 4): mma.sync m16n8k16 with 16 tokens on M and the G heads on
//            N (G = 8 fills the tile, G = 4 half-fills it): S^T = K Q^T, then
//            O^T += V^T P^T with P moved from the accumulator layout to the
//            operand layout by movmatrix.  K/V tiles are 64-column half-tiles
//            with the 128-byte swizzle, so ldmatrix is conflict-free.
//       MMA over an E4M3 cache (fp16 q/out): the same mma.sync, fragments
//            loaded straight from the byte rows and widened in registers by the
//            hardware E4M3 -> f16 conversion.
//       FFMA (G <= 2, or forced): lanes form groups of LPT lanes, a group owns
//            one token at a time, scores use FFMA plus an xor-shuffle reduction.
//     Each warp (MMA) or token group (FFMA) keeps its own running (m, l, acc)
//     in the log2 domain with a lazy rescale (only when the max grows by > 2^8).
//   * end of CTA: groups merge through shared memory into one fp32 partial,
//     which is written to the workspace (or, in the segment-merge modes, merged
//     with the other chunks of its segment through distributed shared memory
//     first, one record per segment); one thread then does
//     fence + atom.add.acq_rel.gpu on the (sequence, KV head) arrival counter.
//     The CTA that sees count == Wtot - 1 is the last arriver: it bulk-copies
//     the records into shared memory, combines them in index order
//     (deterministic), writes out and lse, and resets the counter.  No CTA waits
//     for another CTA's progress outside its own cluster, whose CTAs run
//     together; every other wait is a bounded mbarrier wait on its own loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "fd_common.h"
#include "fd_tcgen05.cuh"

namespace fd {
namespace dev {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr float kLn2 = 0.693147180559945309417f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits give up after ~1 s
constexpr int kCombineBars = 16;  // mbarriers of the combine's copies (one per head of a pass)
constexpr uint32_t kTmemCols = 64;   // tensor-memory columns per CTA (tcgen05 path)
constexpr uint32_t kColS = 0;        // S^T [128 tokens][16 heads]
constexpr uint32_t kColO = 32;       // O^T [128 dims][16 heads]

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` to complete; false after ~1 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - start > kWaitLimitNs) return false;
  }
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue now; and wait until every preceding kernel has finished and its
// memory is visible (a no-op for launches without the PDL attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 3-D tiled TMA load: box at coordinates (c0, c1, c2) of `map` into shared memory.
// Bring one box of a tensor map into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

// Load through L2 only (no L1 line is allocated).
__device__ __forceinline__ int32_t ld_cg_s32(const int32_t* addr) {
  int32_t v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(addr));
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* addr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* addr, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Poll `addr` with acquiring loads until it holds at least `target`; false after
// kCombinerWaitNs (longer than any pipeline wait, so that a CTA whose own waits ran
// out still arrives first).
constexpr uint64_t kCombinerWaitNs = 4 * kWaitLimitNs;
__device__ __forceinline__ bool wait_count_reaches(const uint32_t* addr, uint32_t target) {
  if (ld_acquire_gpu(addr) >= target) return true;
  const uint64_t start = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ld_acquire_gpu(addr) >= target) return true;
    if (global_timer_ns() - start > kCombinerWaitNs) return false;
  }
}
// finish_cta's role for a CTA that does not take part in the combine.
constexpr int kNotCombiner = -1;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
struct Elem;

template <>
struct Elem<__half> {
  static constexpr int kMantissaBits = 11;  // significant bits, implicit one included
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return __half22float2(h);
  }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kMantissaBits = 8;
  // bf16 is the upper half of an fp32 bit pattern: widening is exact.
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& raw, float* f) {
  const float2 a = Elem<T>::to_f2(raw.x), b = Elem<T>::to_f2(raw.y);
  const float2 c = Elem<T>::to_f2(raw.z), d = Elem<T>::to_f2(raw.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}


__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D += A * B for one m16n8k16 tile, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four FP8 E4M3 values (the bytes of x) widened to two f16 pairs with the
// hardware conversion, two values per instruction: lo <- bytes 0 (low half) and 1,
// hi <- bytes 2 and 3.  Every E4M3 value is exact in f16; the codes 0x7F / 0xFF
// (NaN in the format) become NaN.  (An earlier integer widening, prmt + shift +
// mask, kept the ALU pipe 38-50% busy and ran a 32K decode in 17.6 us against 14.6 us
// with this instruction.)
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// Two fp32 values rounded (RN) to one packed 16-bit pair: lo in bits 0-15.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Shared-memory address of 16-byte chunk `ch` (0 .. D/8-1) of token row `row` in a
// tile stored as 64-column half-tiles of `rows` rows with the 128-byte swizzle
// (chunk index XOR row index mod 8, the pattern the TMA writes).
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, int rows, int row, int ch) {
  return base + (uint32_t)((ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// Work item of CTA `cta` in the flattened (sequence, slot, KV head) order.
struct Work {
  int b, kvh, slot, wtot, t0, t1;
  int w, c;       // segment, and chunk within the segment (slot = w * C + c)
  int nrec;       // partial records per query head of sequence b (W_b * rps)
  int rslot;      // this CTA's record slot (slot, or w when segments merge in-cluster)
  int64_t pbase;  // index of the first partial record of sequence b
};

// First partial record of sequence b, and the ready flag of partial `slot` of
// (b, kvh) (fine-grained-waits variant).
__device__ __forceinline__ int64_t rec_base(const Params& p, int b) {
  return (int64_t)(p.unit_base[b] / (p.Hkv * p.C)) * p.rps * p.Hq;
}
__device__ __forceinline__ int flag_index(const Params& p, int b, int kvh, int slot) {
  return p.unit_base[b] + kvh * p.wseg[b] * p.C + slot;
}

// CTA orders within a sequence.  kOrderHeads: KV head fastest, then partial slot.
// kOrderSegment (chunks of a segment merge in a cluster): chunk fastest, then KV
// head, then segment, so that the C chunks of one segment are consecutive (one
// cluster).  kOrderPair (every partial of a (sequence, KV head) in one cluster):
// partial slot fastest, then KV head.
constexpr int kOrderHeads = 0;
constexpr int kOrderSegment = 1;
constexpr int kOrderPair = 2;

__device__ __forceinline__ Work decode_work(const Params& p, int cta, int order) {
  const bool seg = order == kOrderSegment;
  int lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.unit_base[mid] <= cta) lo = mid; else hi = mid;
  }
  Work w;
  w.b = lo;
  const int r = cta - p.unit_base[lo];
  if (order == kOrderHeads) {
    w.kvh = r % p.Hkv;
    w.slot = r / p.Hkv;
    w.w = w.slot / p.C;
    w.c = w.slot - w.w * p.C;
  } else if (order == kOrderPair) {
    const int wc = p.wseg[lo] * p.C;
    w.kvh = r / wc;
    w.slot = r - w.kvh * wc;
    w.w = w.slot / p.C;
    w.c = w.slot - w.w * p.C;
  } else {
    w.c = r % p.C;
    w.kvh = (r / p.C) % p.Hkv;
    w.w = r / (p.C * p.Hkv);
    w.slot = w.w * p.C + w.c;
  }
  w.wtot = p.wseg[lo] * p.C;
  w.nrec = p.wseg[lo] * (seg ? 1 : p.C);
  w.rslot = seg ? w.w : w.slot;
  const int L = p.cu[lo + 1] - p.cu[lo];
  chunk_range(L, p.wseg[lo], p.C, w.slot, p.align, &w.t0, &w.t1);
  w.pbase = rec_base(p, lo);
  return w;
}

// Merge two (max, sum, rounded-weight sum) triples of the log2-domain softmax
// (-inf max = empty).
__device__ __forceinline__ void ml_merge(float& M, float& lam, float& lamr, float m2, float l2,
                                         float lr2) {
  if (m2 == -INFINITY) return;
  if (M == -INFINITY) { M = m2; lam = l2; lamr = lr2; return; }
  if (m2 > M) {
    const float c = ex2(M - m2);
    lam = fmaf(lam, c, l2);
    lamr = fmaf(lamr, c, lr2);
    M = m2;
  } else {
    const float c = ex2(m2 - M);
    lam = fmaf(l2, c, lam);
    lamr = fmaf(lr2, c, lamr);
  }
}

// 1-D bulk copy global -> shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Distributed shared memory of a thread-block cluster: the address of the same
// shared-memory location in CTA `rank` of this cluster, loads from it, and the
// cluster-wide barrier (split into arrive and wait).
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Order this thread's view of generic-proxy global writes before its later
// async-proxy (bulk copy) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Write out[b, h, 4*c4 .. 4*c4+3] = a / lam (zero where lam == 0, i.e. no token; a
// NaN sum, from a NaN in K or V, stays NaN).
template <typename T>
__device__ __forceinline__ void store_out4(T* dst, float4 a, float lam) {
  dst[0] = Elem<T>::from_f(lam != 0.f ? a.x / lam : 0.f);
  dst[1] = Elem<T>::from_f(lam != 0.f ? a.y / lam : 0.f);
  dst[2] = Elem<T>::from_f(lam != 0.f ? a.z / lam : 0.f);
  dst[3] = Elem<T>::from_f(lam != 0.f ? a.w / lam : 0.f);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}


// OnlineSoftmaxCombine of the Wtot partials of (b, kvh) for query heads
// [g0, g0 + ng), from their records in shared memory, head-major
// [ng][wtot][D + 4].  Every thread owns one (head, 4 output dimensions) slice and
// works alone, with no barrier and no shuffle: it reads the partial maxima of its
// head (broadcast loads within the warp) for M, then walks the partials in index
// order, computing coef_w = exp2(m_w - M) and summing coef_w O_w, Lambda =
// sum_w coef_w l_w and Lambda~ = sum_w coef_w l~_w; out = the O sum times 1 /
// Lambda~ (the weights P.V multiplied), lse = M + log Lambda.  Every thread of a
// head computes the same M and Lambdas in the same order, and every sum runs in
// index order, so the result does not depend on the order in which the partials
// arrived.  (Measured on 4 heads x 32 partials: a two-phase form, coefficients by
// one warp per head with shuffle reductions, a barrier, then the weighted sums,
// took ~2200 cycles, most of it in chains of dependent shuffles; this form keeps
// every load of a thread independent.)
template <typename T, int D, int G>
__device__ __forceinline__ void combine_from_smem(const Params& p, int b, int kvh, int wtot,
                                                  int g0, int ng, const float* rec, uint32_t bars,
                                                  uint32_t phase) {
  constexpr int RS = record_floats(D);
  constexpr int Q = D / 4;  // float4 columns per head
  constexpr int U = 8;      // partials in flight per thread
  T* out = reinterpret_cast<T*>(p.out);
  for (int i = threadIdx.x; i < ng * Q; i += kThreads) {
    const int g = i / Q, c4 = i - (i / Q) * Q;
    // This head's records have landed (the copy of each head completes on its own
    // barrier, so the first heads are combined while the later ones still arrive).
    if (!mbar_wait(bars + 8u * (uint32_t)g, phase)) atomicOr(p.status, kStatusTimeout);
    const float* rg = rec + (size_t)g * wtot * RS;
    // M: the largest partial maximum (fmaxf skips NaN maxima; an empty partial has
    // m = -inf).  Four independent running maxima keep the loads in flight.
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    int w = 0;
    for (; w + 4 <= wtot; w += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) m4[u] = fmaxf(m4[u], rg[(size_t)(w + u) * RS + D]);
    }
    for (; w < wtot; ++w) m4[0] = fmaxf(m4[0], rg[(size_t)w * RS + D]);
    const float M = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    const bool none = M == -INFINITY;  // no token in any partial: coefficients 0
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lam = 0.f, lamr = 0.f;
    auto add = [&](const float4& ml, const float4& x) {
      const float c = none ? 0.f : ex2(ml.x - M);
      acc.x = fmaf(c, x.x, acc.x);
      acc.y = fmaf(c, x.y, acc.y);
      acc.z = fmaf(c, x.z, acc.z);
      acc.w = fmaf(c, x.w, acc.w);
      lam = fmaf(c, ml.y, lam);
      lamr = fmaf(c, ml.z, lamr);
    };
    w = 0;
    for (; w + U <= wtot; w += U) {
      float4 ml[U], x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float* r = rg + (size_t)(w + u) * RS;
        ml[u] = *reinterpret_cast<const float4*>(r + D);
        x[u] = *reinterpret_cast<const float4*>(r + 4 * c4);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) add(ml[u], x[u]);
    }
    for (; w < wtot; ++w) {
      const float* r = rg + (size_t)w * RS;
      add(*reinterpret_cast<const float4*>(r + D), *reinterpret_cast<const float4*>(r + 4 * c4));
    }
    const float inv = lamr != 0.f ? 1.f / lamr : 0.f;  // no token: out = 0 (NaN stays NaN)
    T* dst = out + ((int64_t)b * p.Hq + kvh * G + g0 + g) * D + 4 * c4;
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack2<T>(acc.x * inv, acc.y * inv), pack2<T>(acc.z * inv, acc.w * inv));
    if (c4 == 0 && p.lse != nullptr)
      p.lse[(int64_t)b * p.Hq + kvh * G + g0 + g] = lam != 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
  }
}

// Same combine reading the records straight from L2 (for partial counts whose
// records do not fit in shared memory), for query heads [ga, gb) of the pair;
// `coef` holds G * wtot + 3 * G floats (indexed by the head within the pair).
template <typename T, int D, int G>
__device__ __forceinline__ void combine_from_global(const Params& p, int b, int kvh, int wtot,
                                                    int64_t pbase, int ga, int gb, float* coef) {
  constexpr int RS = record_floats(D);
  float* ML = coef + G * wtot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kThreads / 32;
  for (int g = ga + warp; g < gb; g += kWarps) {
    const float* row = p.part + (pbase + (int64_t)(kvh * G + g) * wtot) * RS + D;
    float M = -INFINITY, lam = 0.f, lamr = 0.f;
    for (int w = lane; w < wtot; w += 32) {
      const float4 ml = __ldcg(reinterpret_cast<const float4*>(row + (size_t)w * RS));
      coef[g * wtot + w] = ml.x;
      ml_merge(M, lam, lamr, ml.x, ml.y, ml.z);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, M, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, lam, off);
      const float lr2 = __shfl_xor_sync(0xffffffffu, lamr, off);
      ml_merge(M, lam, lamr, m2, l2, lr2);
    }
    for (int w = lane; w < wtot; w += 32)
      coef[g * wtot + w] = (M == -INFINITY) ? 0.f : ex2(coef[g * wtot + w] - M);
    if (lane == 0) {
      ML[3 * g] = M;
      ML[3 * g + 1] = lam;
      ML[3 * g + 2] = lamr;
    }
  }
  __syncthreads();
  T* out = reinterpret_cast<T*>(p.out);
  for (int v = ga * (D / 4) + tid; v < gb * (D / 4); v += kThreads) {
    const int g = v / (D / 4), c4 = v - (v / (D / 4)) * (D / 4);
    const float4* r =
        reinterpret_cast<const float4*>(p.part + (pbase + (int64_t)(kvh * G + g) * wtot) * RS) + c4;
    const float* cg = coef + g * wtot;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    int w = 0;
    for (; w + 8 <= wtot; w += 8) {
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = __ldcg(r + (size_t)(w + u) * (RS / 4));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float c = cg[w + u];
        a.x = fmaf(c, x[u].x, a.x);
        a.y = fmaf(c, x[u].y, a.y);
        a.z = fmaf(c, x[u].z, a.z);
        a.w = fmaf(c, x[u].w, a.w);
      }
    }
    for (; w < wtot; ++w) {
      const float4 x = __ldcg(r + (size_t)w * (RS / 4));
      const float c = cg[w];
      a.x = fmaf(c, x.x, a.x);
      a.y = fmaf(c, x.y, a.y);
      a.z = fmaf(c, x.z, a.z);
      a.w = fmaf(c, x.w, a.w);
    }
    store_out4<T>(out + ((int64_t)b * p.Hq + kvh * G + g) * D + 4 * c4, a, ML[3 * g + 2]);
  }
  if (ga + tid < gb && p.lse != nullptr) {
    const int g = ga + tid;
    const float M = ML[3 * g], lam = ML[3 * g + 1];
    p.lse[(int64_t)b * p.Hq + kvh * G + g] = lam != 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
  }
}

// Combine all partials of (b, kvh) for query heads [ga, gb) of the pair.  The
// records of as many heads as fit are pulled into shared memory (`smem`,
// `smem_bytes`) in each pass, head j of the pass by bulk copies that complete on
// mbarrier `bars` + 8 j (kCombineBars of them, all at the next phase parity
// `phase`).
template <typename T, int D, int G>
__device__ __forceinline__ void combine_partials(const Params& p, int b, int kvh, int wtot,
                                                 int64_t pbase, int ga, int gb, uint8_t* smem,
                                                 uint32_t smem_bytes, uint32_t bars, uint32_t& phase) {
  constexpr int RS = record_floats(D);
  // Heads per pass: as many heads' records as fit in the shared memory.
  const uint32_t head_bytes = (uint32_t)wtot * RS * 4;
  const int hpp = head_bytes > 0 ? (int)min((uint32_t)min(G, kCombineBars), smem_bytes / head_bytes) : 0;
  if (hpp == 0) {
    combine_from_global<T, D, G>(p, b, kvh, wtot, pbase, ga, gb, reinterpret_cast<float*>(smem));
    return;
  }
  float* rec = reinterpret_cast<float*>(smem);
  for (int g0 = ga; g0 < gb; g0 += hpp) {
    const int ng = min(hpp, gb - g0);
    if (threadIdx.x == 0) {
      fence_proxy_async_global();
      const uint8_t* src = reinterpret_cast<const uint8_t*>(
          p.part + (pbase + (int64_t)(kvh * G + g0) * wtot) * RS);
      const uint32_t dst = smem_addr(smem);
      for (int j = 0; j < ng; ++j) {
        const uint32_t bar = bars + 8u * (uint32_t)j, h0 = (uint32_t)j * head_bytes;
        mbar_arrive_expect_tx(bar, head_bytes);
        for (uint32_t off = 0; off < head_bytes; off += 32768u)
          bulk_load(dst + h0 + off, src + h0 + off, min(32768u, head_bytes - off), bar);
      }
    }
    combine_from_smem<T, D, G>(p, b, kvh, wtot, g0, ng, rec, bars, phase);
    phase ^= 1u;
    __syncthreads();  // the next pass overwrites the records
  }
}

// Fine-grained waits (the pages' "combine each partial as it arrives"): the CTA
// of slot 0 of (b, kvh) polls the ready flags of all Wtot partials and folds every
// batch that has arrived into a running (M, Lambda, O), in arrival order.  The
// whole grid is co-resident (cooperative launch), so every producer can finish;
// the poll is still bounded and reports a timeout through the status word.
// `sm` provides G * (D + 4) + 2 * wtot + G * wtot + 2 floats of scratch.
template <typename T, int D, int G>
__device__ __forceinline__ void combine_as_arrived(const Params& p, const Work& wk, float* sm) {
  constexpr int RS = record_floats(D);
  const int wtot = wk.wtot;
  float* run_O = sm;                       // [G][D]
  float* run_M = run_O + G * D;            // [G]
  float* run_L = run_M + G;                // [G]
  float* run_Lr = run_L + G;               // [G] rounded-weight sums
  float* coef = run_Lr + G;                // [G][wtot] (this batch)
  float* scl = coef + G * wtot;            // [G]
  int* ready = reinterpret_cast<int*>(scl + G);  // [wtot] slots of this batch
  int* done = ready + wtot;                // [wtot]
  int* ctl = done + wtot;                  // [0] batch size, [1] stop
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kThreads / 32;
  const int fbase = flag_index(p, wk.b, wk.kvh, 0);  // flag of slot w: fbase + w
  for (int i = tid; i < G * D; i += kThreads) run_O[i] = 0.f;
  for (int g = tid; g < G; g += kThreads) { run_M[g] = -INFINITY; run_L[g] = 0.f; run_Lr[g] = 0.f; }
  for (int w = tid; w < wtot; w += kThreads) done[w] = 0;
  if (tid == 0) ctl[1] = 0;
  __syncthreads();
  const uint64_t start = global_timer_ns();
  int merged = 0;
  while (merged < wtot) {
    if (tid == 0) ctl[0] = 0;
    __syncthreads();
    for (int w = tid; w < wtot; w += kThreads) {
      if (!done[w] && (w == wk.slot || ld_acquire_gpu(p.flags + fbase + w) != 0u)) {
        done[w] = 1;
        ready[atomicAdd(&ctl[0], 1)] = w;
      }
    }
    if (tid == 0 && global_timer_ns() - start > kWaitLimitNs) ctl[1] = 1;
    __syncthreads();
    const int n = ctl[0];
    if (n == 0) {
      if (ctl[1]) {
        if (tid == 0) atomicOr(p.status, kStatusTimeout);
        break;
      }
      continue;
    }
    // (M, Lambda) update per head for this batch.
    for (int g = warp; g < G; g += kWarps) {
      const int64_t row = wk.pbase + (int64_t)(wk.kvh * G + g) * wtot;
      float mx = -INFINITY;
      for (int i = lane; i < n; i += 32)
        mx = fmaxf(mx, __ldcg(p.part + (row + ready[i]) * RS + D));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float Mold = run_M[g];
      const float Mnew = fmaxf(Mold, mx);
      float lam = 0.f, lamr = 0.f;
      for (int i = lane; i < n; i += 32) {
        const float4 ml = __ldcg(reinterpret_cast<const float4*>(p.part + (row + ready[i]) * RS + D));
        const float c = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - Mnew);
        coef[g * wtot + i] = c;
        lam = fmaf(c, ml.y, lam);
        lamr = fmaf(c, ml.z, lamr);
      }
      lam = warp_sum(lam);
      lamr = warp_sum(lamr);
      if (lane == 0) {
        const float sc = (Mold == -INFINITY) ? 0.f : ex2(Mold - Mnew);
        scl[g] = sc;
        run_L[g] = fmaf(run_L[g], sc, lam);
        run_Lr[g] = fmaf(run_Lr[g], sc, lamr);
        run_M[g] = Mnew;
      }
    }
    __syncthreads();
    for (int v = tid; v < G * (D / 4); v += kThreads) {
      const int g = v / (D / 4), c4 = v - (v / (D / 4)) * (D / 4);
      const int64_t row = wk.pbase + (int64_t)(wk.kvh * G + g) * wtot;
      float4 a = reinterpret_cast<float4*>(run_O + g * D)[c4];
      const float sc = scl[g];
      a.x *= sc; a.y *= sc; a.z *= sc; a.w *= sc;
      for (int i = 0; i < n; ++i) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(p.part + (row + ready[i]) * RS) + c4);
        const float c = coef[g * wtot + i];
        a.x = fmaf(c, x.x, a.x);
        a.y = fmaf(c, x.y, a.y);
        a.z = fmaf(c, x.z, a.z);
        a.w = fmaf(c, x.w, a.w);
      }
      reinterpret_cast<float4*>(run_O + g * D)[c4] = a;
    }
    merged += n;
    __syncthreads();
  }
  // Flags go back to zero for the next decode (the ones that were set).
  for (int w = tid; w < wtot; w += kThreads)
    if (done[w] && w != wk.slot) p.flags[fbase + w] = 0u;
  if (merged < wtot) return;  // timed out: status is set, out is not written
  T* out = reinterpret_cast<T*>(p.out);
  for (int v = tid; v < G * (D / 4); v += kThreads) {
    const int g = v / (D / 4), c4 = v - (v / (D / 4)) * (D / 4);
    store_out4<T>(out + ((int64_t)wk.b * p.Hq + wk.kvh * G + g) * D + 4 * c4,
                  reinterpret_cast<float4*>(run_O + g * D)[c4], run_Lr[g]);
  }
  if (tid < G && p.lse != nullptr) {
    const float M = run_M[tid], lam = run_L[tid];
    p.lse[(int64_t)wk.b * p.Hq + wk.kvh * G + tid] = lam != 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
  }
}

// Segment merge inside a thread-block cluster (the C chunk CTAs of one segment):
// every CTA holds its chunk record in shared memory (`crec`, [G][D + 4]); after a
// cluster barrier each CTA reads all C records through distributed shared memory
// and writes its share of the columns of the segment's record (fixed chunk
// order; CTA 0 also writes M and the two Lambdas).  Ends with this CTA's arrival
// at the closing cluster barrier; the caller waits on it before the CTA exits, so
// no CTA leaves while another still reads its shared memory.  `cf` is scratch for
// G * (C + 3) floats.
template <int D, int G>
__device__ __forceinline__ void merge_segment(const Params& p, const Work& wk, const float* crec,
                                              float* cf) {
  constexpr int RS = record_floats(D);
  const int tid = threadIdx.x, C = p.C;
  cluster_arrive();
  cluster_wait();  // every chunk record of the segment is in place
  const uint32_t crec_a = smem_addr(crec);
  if (tid < G) {
    const uint32_t ml_a = crec_a + (uint32_t)(tid * RS + D) * 4u;
    float M = -INFINITY;
    for (int j = 0; j < C; ++j) M = fmaxf(M, ld_cluster_f2(cluster_map(ml_a, j)).x);
    float lam = 0.f, lamr = 0.f;
    for (int j = 0; j < C; ++j) {
      const float4 ml = ld_cluster_f4(cluster_map(ml_a, j));
      const float f = (M == -INFINITY) ? 0.f : ex2(ml.x - M);  // an empty chunk has m = -inf
      cf[tid * C + j] = f;
      lam = fmaf(f, ml.y, lam);
      lamr = fmaf(f, ml.z, lamr);
    }
    cf[G * C + tid] = M;
    cf[G * C + G + tid] = lam;
    cf[G * C + 2 * G + tid] = lamr;
  }
  __syncthreads();
  constexpr int Q = D / 4;
  const int lo4 = wk.c * Q / C, n4 = (wk.c + 1) * Q / C - lo4;
  const int64_t rec0 = wk.pbase + (int64_t)(wk.kvh * G) * wk.nrec + wk.w;  // head g: + g * nrec
  for (int i = tid; i < G * n4; i += kThreads) {
    const int g = i / n4, c4 = lo4 + (i - (i / n4) * n4);
    const uint32_t src = crec_a + (uint32_t)(g * RS + 4 * c4) * 4u;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < C; ++j) {
      const float4 x = ld_cluster_f4(cluster_map(src, j));
      const float f = cf[g * C + j];
      acc.x = fmaf(f, x.x, acc.x);
      acc.y = fmaf(f, x.y, acc.y);
      acc.z = fmaf(f, x.z, acc.z);
      acc.w = fmaf(f, x.w, acc.w);
    }
    __stcg(reinterpret_cast<float4*>(p.part + (rec0 + (int64_t)g * wk.nrec) * RS) + c4, acc);
  }
  if (wk.c == 0 && tid < G)
    __stcg(reinterpret_cast<float4*>(p.part + (rec0 + (int64_t)tid * wk.nrec) * RS + D),
           make_float4(cf[G * C + tid], cf[G * C + G + tid], cf[G * C + 2 * G + tid], 0.f));
  cluster_arrive();  // done reading the other CTAs' shared memory
}

// OnlineSoftmaxCombine of all Wtot partials of (b, kvh) inside one thread-block
// cluster (the Wtot CTAs of the pair, cluster rank = partial slot): every CTA holds
// its record in shared memory (`crec`, [G][D + 4]); after a cluster barrier each CTA
// reads the (m, l, l~) of all records through distributed shared memory, then
// combines its share of the G x D output columns from all Wtot records, in slot
// order, and writes out (CTA 0 also writes lse).  No global records, no counter.
// A closing cluster barrier keeps every CTA alive until no peer reads its shared
// memory.  `cf` is scratch for G * (Wtot + 3) floats.
template <typename T, int D, int G>
__device__ __forceinline__ void combine_in_cluster(const Params& p, const Work& wk, const float* crec,
                                                   float* cf) {
  constexpr int RS = record_floats(D);
  constexpr int kMaxCluster = 16;
  const int tid = threadIdx.x, CS = wk.wtot;
  cluster_arrive();
  cluster_wait();  // every record of the pair is in place
  const uint32_t crec_a = smem_addr(crec);
  if (tid < G) {
    const uint32_t ml_a = crec_a + (uint32_t)(tid * RS + D) * 4u;
    float4 ml[kMaxCluster];
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j)
      if (j < CS) ml[j] = ld_cluster_f4(cluster_map(ml_a, j));
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j)
      if (j < CS) M = fmaxf(M, ml[j].x);
    float lam = 0.f, lamr = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
      if (j < CS) {
        const float f = (M == -INFINITY) ? 0.f : ex2(ml[j].x - M);  // an empty partial has m = -inf
        cf[tid * CS + j] = f;
        lam = fmaf(f, ml[j].y, lam);
        lamr = fmaf(f, ml[j].z, lamr);
      }
    }
    cf[G * CS + tid] = M;
    cf[G * CS + G + tid] = lam;
    cf[G * CS + 2 * G + tid] = lamr;
  }
  __syncthreads();
  constexpr int Q = D / 4;
  const int n = G * Q, lo = wk.slot * n / CS, hi = (wk.slot + 1) * n / CS;
  T* out = reinterpret_cast<T*>(p.out);
  for (int i = lo + tid; i < hi; i += kThreads) {
    const int g = i / Q, c4 = i - (i / Q) * Q;
    const uint32_t src = crec_a + (uint32_t)(g * RS + 4 * c4) * 4u;
    float4 x[kMaxCluster];
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j)
      if (j < CS) x[j] = ld_cluster_f4(cluster_map(src, j));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
      if (j < CS) {
        const float f = cf[g * CS + j];
        acc.x = fmaf(f, x[j].x, acc.x);
        acc.y = fmaf(f, x[j].y, acc.y);
        acc.z = fmaf(f, x[j].z, acc.z);
        acc.w = fmaf(f, x[j].w, acc.w);
      }
    }
    store_out4<T>(out + ((int64_t)wk.b * p.Hq + wk.kvh * G + g) * D + 4 * c4, acc,
                  cf[G * CS + 2 * G + g]);
  }
  if (wk.slot == 0 && tid < G && p.lse != nullptr) {
    const float M = cf[G * CS + tid], lam = cf[G * CS + G + tid];
    p.lse[(int64_t)wk.b * p.Hq + wk.kvh * G + tid] = lam != 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
  }
  cluster_arrive();  // done reading the other CTAs' shared memory
  cluster_wait();
}

// Merge NGRP running states (sm_acc [NGRP][G][D], sm_m / sm_l / sm_lr [NGRP][G],
// all in shared memory; sm_lr sums the rounded weights P.V used) into this CTA's
// partial; then either finish directly (a single
// partial), or publish the partial (merged per segment inside the cluster when
// rps == 1), arrive, and combine if this CTA arrived last.  An `aborted` CTA (its
// pipeline timed out; the status word says so) contributes an empty partial so
// that its cluster and its (b, kvh) counter still complete.
template <typename T, int D, int G, int NGRP, int MODE, bool SEG, bool PAIR>
__device__ __forceinline__ void finish_cta(const Params& p, const Work& wk, float* sm_acc,
                                           int& sm_last, bool aborted, uint8_t* combine_smem,
                                           uint32_t combine_bytes, uint32_t combine_bars) {
  float* sm_m = sm_acc + NGRP * G * D;  // [NGRP][G]
  float* sm_l = sm_m + NGRP * G;        // [NGRP][G]
  float* sm_lr = sm_l + NGRP * G;       // [NGRP][G]
  float* sm_fac = sm_lr + NGRP * G;     // [NGRP][G]
  float* sm_ML = sm_fac + NGRP * G;     // [G][3]: M, Lambda, Lambda~
  const int tid = threadIdx.x;
  if (tid < G) {
    const int g = tid;
    float M = -INFINITY;
    for (int q = 0; q < NGRP; ++q) M = fmaxf(M, sm_m[q * G + g]);
    float lam = 0.f, lamr = 0.f;
    for (int q = 0; q < NGRP; ++q) {
      const float f = (M == -INFINITY) ? 0.f : ex2(sm_m[q * G + g] - M);
      sm_fac[q * G + g] = f;
      lam = fmaf(sm_l[q * G + g], f, lam);
      lamr = fmaf(sm_lr[q * G + g], f, lamr);
    }
    sm_ML[3 * g] = aborted ? -INFINITY : M;
    sm_ML[3 * g + 1] = aborted ? 0.f : lam;
    sm_ML[3 * g + 2] = aborted ? 0.f : lamr;
  }
  __syncthreads();

  const int h0 = wk.kvh * G;
  if ((MODE == 0 || MODE == 3) && wk.wtot == 1) {
    // A single partial is already the answer: normalise and store.
    T* out = reinterpret_cast<T*>(p.out);
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int g = idx / D, dim = idx - (idx / D) * D;
      float a = 0.f;
#pragma unroll 4
      for (int q = 0; q < NGRP; ++q) a = fmaf(sm_acc[(q * G + g) * D + dim], sm_fac[q * G + g], a);
      const float lamr = sm_ML[3 * g + 2];
      out[((int64_t)wk.b * p.Hq + h0 + g) * D + dim] = Elem<T>::from_f(lamr != 0.f ? a / lamr : 0.f);
    }
    if (tid < G && p.lse != nullptr) {
      const float M = sm_ML[3 * tid], lam = sm_ML[3 * tid + 1];
      p.lse[(int64_t)wk.b * p.Hq + h0 + tid] = lam != 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
    }
    return;
  }

  // Publish this CTA's partial record (O unnormalised w.r.t. M, then M, Lambda):
  // to global memory, or to `crec` at the end of the ring for the segment merge.
  constexpr int RS = record_floats(D);
  constexpr bool merge_seg = SEG || PAIR;  // the record goes to shared memory
  static_assert(!SEG || MODE == 0 || MODE == 1, "segment merge: fused or split-only kernels");
  static_assert(!PAIR || MODE == 0, "pair clusters: fused kernel");
  const uint32_t crec_bytes = merge_seg ? (uint32_t)(G * RS * 4) : 0u;
  float* crec = reinterpret_cast<float*>(combine_smem + combine_bytes - G * RS * 4);
  for (int idx = tid; idx < G * D / 4; idx += kThreads) {
    const int g = idx / (D / 4), c4 = idx - (idx / (D / 4)) * (D / 4);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int q = 0; q < NGRP; ++q) {
      const float4 x = reinterpret_cast<const float4*>(sm_acc + (q * G + g) * D)[c4];
      const float f = sm_fac[q * G + g];
      a.x = fmaf(x.x, f, a.x);
      a.y = fmaf(x.y, f, a.y);
      a.z = fmaf(x.z, f, a.z);
      a.w = fmaf(x.w, f, a.w);
    }
    if (aborted) a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (merge_seg) {
      reinterpret_cast<float4*>(crec + g * RS)[c4] = a;
    } else {
      const int64_t pidx = wk.pbase + (int64_t)(h0 + g) * wk.nrec + wk.rslot;
      __stcg(reinterpret_cast<float4*>(p.part + pidx * RS) + c4, a);
    }
  }
  if (tid < G) {
    const float4 ml = make_float4(sm_ML[3 * tid], sm_ML[3 * tid + 1], sm_ML[3 * tid + 2], 0.f);
    if (merge_seg) {
      *reinterpret_cast<float4*>(crec + tid * RS + D) = ml;
    } else {
      const int64_t pidx = wk.pbase + (int64_t)(h0 + tid) * wk.nrec + wk.rslot;
      __stcg(reinterpret_cast<float4*>(p.part + pidx * RS + D), ml);
    }
  }
  if constexpr (PAIR) {
    combine_in_cluster<T, D, G>(p, wk, crec, sm_acc);
    return;
  }
  if (merge_seg) merge_segment<D, G>(p, wk, crec, sm_acc);
  if (MODE == 1) {
    if (merge_seg) cluster_wait();
    return;
  }
  if (MODE == 3) {
    __syncthreads();
    if (wk.slot != 0) {
      const bool dropped = p.test_hook == kHookDropFlag && wk.b == 0 && wk.kvh == 0 && wk.slot == 1;
      if (tid == 0 && !dropped) st_release_gpu(p.flags + flag_index(p, wk.b, wk.kvh, wk.slot), 1u);
      return;
    }
    combine_as_arrived<T, D, G>(p, wk, reinterpret_cast<float*>(combine_smem));
    return;
  }

  // Arrival: the CTA's stores are ordered before thread 0's release by the barrier
  // (release is cumulative); the acquiring RMW makes every earlier CTA's record
  // visible to the last arriver, whose threads are ordered after it by the barrier.
  // The last `nc` arrivals share the combine: arrival r before the last (r = 0 is
  // the last) combines query heads [r G / nc, (r + 1) G / nc) once an acquiring load
  // of the counter reads Wtot (the release sequence of the arrivals' RMWs makes
  // every record visible to it).  Only a plan whose whole grid is resident at once
  // has nc > 1, so the arrivals it waits for always run.
  __syncthreads();
  uint32_t* cnt = p.counters + (int64_t)wk.b * p.Hkv + wk.kvh;
  int nc = p.combiners;
  while (nc > wk.wtot) nc >>= 1;  // a power of two dividing G
  const bool drop_arrival =
      p.test_hook == kHookDropArrival && wk.b == 0 && wk.kvh == 0 && wk.slot == 1;
  if (tid == 0 && drop_arrival) sm_last = kNotCombiner;
  if (tid == 0 && !drop_arrival) {
    const uint32_t old = atom_add_acq_rel_gpu(cnt, 1u);
    if (old >= (uint32_t)wk.wtot) atomicOr(p.status, kStatusCounter);
    const int r = wk.wtot - 1 - (int)min(old, (uint32_t)wk.wtot);
    int role = (r >= 0 && r < nc) ? r : kNotCombiner;
    if (role > 0 && !wait_count_reaches(cnt, (uint32_t)wk.wtot)) {
      atomicOr(p.status, kStatusTimeout);
      role = kNotCombiner;  // the workspace needs fd_workspace_init after this
    }
    if (role >= 0) {  // only a combining CTA pays for its copy barriers
      for (int j = 0; j < kCombineBars; ++j) mbar_init(combine_bars + 8u * j, 1);
      fence_mbar_init();
    }
    sm_last = role;
  }
  __syncthreads();
  const int role = sm_last;
  if (role >= 0) {
    // The records end before `crec`, which other CTAs of the cluster may still read.
    uint32_t phase = 0;
    const int hpc = G / nc;
    combine_partials<T, D, G>(p, wk.b, wk.kvh, wk.nrec, wk.pbase, role * hpc, (role + 1) * hpc,
                              combine_smem, combine_bytes - crec_bytes, combine_bars, phase);
    if (tid == 0) {
      // The counter returns to zero once every combiner has read Wtot from it.
      if (nc == 1 || atomicAdd(cnt, 1u) == (uint32_t)(wk.wtot + nc - 1)) *cnt = 0u;
    }
  }
  if (merge_seg) cluster_wait();
}

// MODE 0: fused split + last-arriver combine.  MODE 1: split only (partials).
// MODE 3: fused split + fine-grained waits.  MODE 4 / 5: MODE 0 / 1 with each
// segment's chunk partials merged inside a thread-block cluster (rps == 1).
// MODE 6: fused, every partial of a (sequence, KV head) in one thread-block cluster
// that combines them through distributed shared memory.
// CPS: resident CTAs per SM the kernel is built for; 3 (kShallowCtasPerSm) gives it
// the 64 KB ring of plans of many short CTAs (mma.sync path, fused), else 2.
template <typename T, int D, int G, int PATH, int MODE, int CPS = 2>
__global__ void __launch_bounds__(kThreads, CPS) fd_split_kernel(const __grid_constant__ Params p) {
  constexpr bool kSeg = MODE == 4 || MODE == 5;
  constexpr bool kPair = MODE == 6;
  constexpr int kMode = kSeg ? MODE - 4 : kPair ? 0 : MODE;
  constexpr int TILE = tile_for(PATH);
  constexpr int LPT = loads_per_tile(PATH);       // ring slots per tile (2: K and V apart)
  constexpr int NSLOT = ring_slots_for(PATH, D, CPS);  // ring slots
  constexpr int BOXC = box_cols_for(PATH, D);   // columns per TMA box
  constexpr int NBOX = D / BOXC;                // boxes per tensor per stage
  constexpr int KVES = kv_elem_bytes(PATH);     // bytes per stored K/V element
  constexpr uint32_t kRowsBytes = TILE * D * KVES;  // one tile of K (or V) rows
  constexpr uint32_t kSlotBytes = (2 / LPT) * kRowsBytes;  // K rows then V rows, or one of them
  constexpr uint32_t kRing = NSLOT * kSlotBytes;
  constexpr uint32_t kExtra = extra_bytes_for(PATH);
  static_assert(NSLOT >= 2 && kRowsBytes % 1024 == 0, "slots hold whole swizzle atoms");
  static_assert((2 * NSLOT + 5 + kCombineBars) * 8 + 1024 <= kRingMetaBytes, "ring metadata must fit");
  static_assert(kRing == ring_bytes_for(PATH, D, CPS), "ring layout");
  constexpr int NGRP_FFMA = kConsumerWarps * (32 / ((G * D > 512) ? 16 : 8));
  constexpr int NGRP = PATH == kPathUmma ? 1 : is_mma(PATH) ? kConsumerWarps : NGRP_FFMA;
  static_assert(PATH == kPathFfma || G >= 4, "the MMA path needs G >= 4 heads on N");
  static_assert(NGRP * G * D * 4 + 4 * NGRP * G * 4 + 3 * G * 4 + G * record_floats(D) * 4 <= kRing,
                "group merge and the segment-merge record must fit in the ring");

  // 1024-byte aligned ring: the 128-byte swizzle pattern repeats every 1024 bytes.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRing + kExtra);
  int& sm_abort = *reinterpret_cast<int*>(bars + 2 * NSLOT + 1);
  int& sm_last = *(reinterpret_cast<int*>(bars + 2 * NSLOT + 1) + 1);
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + NSLOT + s); };
  // tcgen05 path: S^T ready, every MMA done, and the tensor-memory base address.
  const uint32_t bar_s = smem_addr(bars + 2 * NSLOT + 2);
  const uint32_t bar_o = smem_addr(bars + 2 * NSLOT + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NSLOT + 4);
  const uint32_t combine_bars = smem_addr(bars + 2 * NSLOT + 5);  // kCombineBars of them

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  // Prologue that touches no global memory: it may overlap the previous kernel.
  const Work wk = decode_work(p, blockIdx.x, kSeg ? kOrderSegment : kPair ? kOrderPair : kOrderHeads);
  const int ntiles = (wk.t1 - wk.t0 + TILE - 1) / TILE;
  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full_bar(s), 1);
      // Released by every consumer warp, or by one tcgen05 commit.
      mbar_init(empty_bar(s), PATH == kPathUmma ? 1 : kConsumerWarps);
    }
    if (PATH == kPathUmma) {
      mbar_init(bar_s, 1);
      mbar_init(bar_o, 1);
    }
    fence_mbar_init();
    sm_abort = 0;
  }
  if constexpr (PATH == kPathUmma) {
    // 64 tensor-memory columns: S^T at 0..15, O^T at 32..47 (two CTAs per SM use 128
    // of the 512, so the allocation never waits).
    if (warp == 0) {
      tc::tmem_alloc(smem_addr(tmem_slot), kTmemCols);
      tc::tmem_relinquish();
    }
  }
  if (warp == kConsumerWarps && lane == 0 && ntiles > 0) {
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    // Warm L2 with the first tiles of the chunk while the previous kernel drains
    // (its combine tail leaves HBM idle).  An L2 prefetch hands no data to this
    // SM, and L2 is where every global write becomes visible, so it cannot expose
    // K/V that the previous kernel is still writing.  CTAs past the first wave,
    // which start after the previous kernel, skip it.
    if ((int)blockIdx.x < p.prefetch_ctas) {
      const int npf = min(ntiles, kL2PrefetchTokens / TILE);
      if (p.block_table == nullptr) {
        const int row0 = p.cu[wk.b] + wk.t0;
        for (int kt = 0; kt < npf; ++kt) {
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx) {
            tma_prefetch_l2_3d(&p.tm_k, bx * BOXC, wk.kvh, row0 + kt * TILE);
            tma_prefetch_l2_3d(&p.tm_v, bx * BOXC, wk.kvh, row0 + kt * TILE);
          }
        }
      } else if (p.box_rows == TILE) {
        // Paged (pages of at least one tile; smaller pages would need many small
        // prefetches, which measured slower): the block table may itself be written
        // by the previous kernel, so these entries are only a guess (read through
        // L2, leaving no L1 line that the loads after the wait could hit).  A wrong
        // page costs bandwidth, never
        // correctness: the loads re-read the table after the wait, and a prefetch
        // outside the pool fetches nothing.
        const int32_t* bt = p.block_table + (int64_t)wk.b * p.bt_stride;
        const int last_pg = (p.cu[wk.b + 1] - p.cu[wk.b] - 1) >> p.page_shift;
        for (int kt = 0; kt < npf; ++kt) {
          const int a = wk.t0 + kt * TILE;
          for (int r = 0; r < TILE; r += p.box_rows) {
            const int pg = ld_cg_s32(bt + min((a + r) >> p.page_shift, last_pg));
            if (pg < 0 || pg > (0x3fffffff >> p.page_shift)) continue;
            const int row = pg * (1 << p.page_shift) + ((a + r) & ((1 << p.page_shift) - 1));
#pragma unroll
            for (int bx = 0; bx < NBOX; ++bx) {
              tma_prefetch_l2_3d(&p.tm_k, bx * BOXC, wk.kvh, row);
              tma_prefetch_l2_3d(&p.tm_v, bx * BOXC, wk.kvh, row);
            }
          }
        }
      }
    }
  }
  pdl_wait();  // q, K, V, the workspace and out may come from earlier kernels
  if constexpr (PATH == kPathUmma) tc::fence_before_sync();
  __syncthreads();

  float* sm_acc = reinterpret_cast<float*>(smem);  // [NGRP][G][D] after the ring drains
  float* sm_m = sm_acc + NGRP * G * D;
  float* sm_l = sm_m + NGRP * G;
  float* sm_lr = sm_l + NGRP * G;  // sums of the rounded weights P.V used

  if (warp == kConsumerWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && ntiles > 0) {
      const uint64_t policy = l2_evict_first_policy();
      const int row0 = p.cu[wk.b] + wk.t0;
      // Load j goes to slot j mod NSLOT.  One load per tile: its K rows, then its V
      // rows; two loads per tile (tcgen05 path): K rows (j even), then V rows.
      const int nload = ntiles * LPT;
      int j = 0;
      for (; j < nload; ++j) {
        const int s = j % NSLOT, kt = j / LPT;
        if (j >= NSLOT && !mbar_wait(empty_bar(s), ((j / NSLOT) - 1) & 1)) {
          atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
          break;
        }
        if (*(volatile int*)&sm_abort) break;
        if (p.test_hook == kHookSkipTile && kt == 1 && wk.b == 0 && wk.kvh == 0 && wk.slot == 0)
          continue;  // test hook: this tile is never loaded
        const uint32_t dst = smem_addr(smem + (size_t)s * kSlotBytes);
        const int h0 = LPT == 2 ? (j & 1) : 0, h1 = LPT == 2 ? (j & 1) + 1 : 2;
        mbar_arrive_expect_tx(full_bar(s), kSlotBytes);
        if (p.block_table == nullptr) {
#pragma unroll
          for (int h = h0; h < h1; ++h) {  // K rows, then V rows
#pragma unroll
            for (int bx = 0; bx < NBOX; ++bx)
              tma_load_3d(dst + (h - h0) * kRowsBytes + bx * (TILE * BOXC * KVES),
                          h ? &p.tm_v : &p.tm_k, bx * BOXC, wk.kvh, row0 + kt * TILE, full_bar(s),
                          policy);
          }
        } else {
          // Paged: one box per page piece of the tile.  Tiles start on multiples of
          // the tile size, so each box stays inside one page; boxes past the end of
          // the sequence reload its last page (their rows are masked).
          const int32_t* bt = p.block_table + (int64_t)wk.b * p.bt_stride;
          const int last_pg = (p.cu[wk.b + 1] - p.cu[wk.b] - 1) >> p.page_shift;
          const int a = wk.t0 + kt * TILE;
          for (int r = 0; r < TILE; r += p.box_rows) {
            const int pg = min((a + r) >> p.page_shift, last_pg);
            const int row = __ldg(bt + pg) * (1 << p.page_shift) + ((a + r) & ((1 << p.page_shift) - 1));
#pragma unroll
            for (int h = h0; h < h1; ++h) {  // K rows, then V rows
#pragma unroll
              for (int bx = 0; bx < NBOX; ++bx)
                tma_load_3d(dst + (h - h0) * kRowsBytes + bx * (TILE * BOXC * KVES) + r * BOXC * KVES,
                            h ? &p.tm_v : &p.tm_k, bx * BOXC, wk.kvh, row, full_bar(s), policy);
            }
          }
        }
      }
      // Every load issued must land before shared memory is reused or released.
      for (int t = (j > NSLOT ? j - NSLOT : 0); t < j; ++t) {
        if (!mbar_wait(full_bar(t % NSLOT), (t / NSLOT) & 1)) atomicOr(p.status, kStatusTimeout);
      }
    }
    __syncthreads();
  } else if constexpr (PATH == kPathUmma) {
    // ---------------- tcgen05 consumers ----------------
    // Thread tid (0..127) owns row tid of S^T (token tid of the tile) and of O^T
    // (head dimension tid), i.e. TMEM lane tid, which its warp's quarter reaches.
    // Thread 0 also issues every MMA.  The running max m is per head and uniform
    // across the CTA; l and l~ are per-thread partial sums over its tokens.
    static_assert(D == 128 && (G == 4 || G == 8 || G == 16), "tcgen05 path: d = 128, G in {4, 8, 16}");
    constexpr int NP = 16;  // MMA N: the G heads, padded with zero rows of Q
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdS = tc::idesc_f16(kBf16, false, false, 128, NP);  // K, Q: K-major
    constexpr uint32_t kIdO = tc::idesc_f16(kBf16, true, true, 128, NP);    // V^T, P^T: MN-major
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quarter
    uint8_t* qs = smem + kRing;        // Q: 16 rows x 128, two 64-column 128-byte-swizzled halves
    uint8_t* ps = qs + 4096;           // P^T: 128 token rows x 16 heads, 32-byte swizzle
    float* wmax = reinterpret_cast<float*>(qs + 8192);  // [4 warps][16] per-warp tile maxima
    // bf16: the residuals of the rounded weights, P^T's second part (same layout); P.V
    // takes hi + lo, 16 significant bits (a weight rounded once to bf16 is off by up
    // to 2^-9 of itself, enough over a few tokens to move out past the tolerance).
    uint8_t* ps_lo = qs + 9216;
    const uint32_t qs_a = smem_addr(qs), ps_a = smem_addr(ps), ps_lo_a = smem_addr(ps_lo);

    // Q into shared memory (zero rows for the padding heads).
    for (int c = tid; c < NP * (D / 8); c += 4 * 32) {
      const int r = c / (D / 8), ch = c - r * (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < G)
        v = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.q) +
                                             ((int64_t)wk.b * p.Hq + wk.kvh * G + r) * D + ch * 8);
      *reinterpret_cast<uint4*>(qs + (ch >> 3) * 2048 + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
    }
    tc::fence_proxy_async_smem();
    tc::named_sync(1, 4 * 32);

    // S^T(kt) = K(kt) Q^T into columns kColS; releases K's slot when done.
    auto issue_s = [&](int kt) -> bool {
      const int jl = kt * 2, s = jl % NSLOT;
      if (!mbar_wait(full_bar(s), (jl / NSLOT) & 1)) return false;
      tc::fence_after_sync();
      const uint32_t ka = smem_addr(smem + (size_t)s * kSlotBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_f16_ss(tmem + kColS,
                       tc::smem_desc(ka + (kk >> 2) * (TILE * 128) + (kk & 3) * 32, 16, 1024,
                                     tc::kSwizzle128B),
                       tc::smem_desc(qs_a + (kk >> 2) * (NP * 128) + (kk & 3) * 32, 16, 1024,
                                     tc::kSwizzle128B),
                       kIdS, kk > 0);
      tc::commit(empty_bar(s));
      tc::commit(bar_s);
      return true;
    };
    // O^T += V(kt)^T P^T into columns kColO; releases V's slot when done.
    auto issue_pv = [&](int kt) -> bool {
      const int jl = kt * 2 + 1, s = jl % NSLOT;
      if (!mbar_wait(full_bar(s), (jl / NSLOT) & 1)) return false;
      tc::fence_after_sync();
      const uint32_t va = smem_addr(smem + (size_t)s * kSlotBytes);
#pragma unroll
      for (int kk = 0; kk < TILE / 16; ++kk)
        tc::mma_f16_ss(tmem + kColO,
                       tc::smem_desc(va + kk * 2048, TILE * 128, 1024, tc::kSwizzle128B),
                       tc::smem_desc(ps_a + kk * 512, 16, 256, tc::kSwizzle32B),
                       kIdO, (kt > 0 || kk > 0) ? 1u : 0u);
      if constexpr (kBf16) {
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          tc::mma_f16_ss(tmem + kColO,
                         tc::smem_desc(va + kk * 2048, TILE * 128, 1024, tc::kSwizzle128B),
                         tc::smem_desc(ps_lo_a + kk * 512, 16, 256, tc::kSwizzle32B), kIdO, 1u);
      }
      tc::commit(empty_bar(s));
      return true;
    };
    auto give_up = [&]() {  // thread 0: a load never arrived
      atomicOr(p.status, kStatusTimeout);
      *(volatile int*)&sm_abort = 1;
    };

    float m_run[G], l_ex[G], l_rd[G];
#pragma unroll
    for (int g = 0; g < G; ++g) { m_run[g] = -INFINITY; l_ex[g] = 0.f; l_rd[g] = 0.f; }
    const float scale = p.scale_log2;
    if (tid == 0 && ntiles > 0 && !issue_s(0)) {
      give_up();
      mbar_arrive(bar_s);
    }
    __syncwarp();
    for (int kt = 0; kt < ntiles; ++kt) {
      const bool ok = mbar_wait(bar_s, kt & 1);
      tc::fence_after_sync();
      float x[16];
      tc::ld16(tmem + trow + kColS, x);
      tc::wait_ld();
      const int ntok = min(TILE, wk.t1 - (wk.t0 + kt * TILE));
      const bool valid = tid < ntok;
      bool need = false;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        x[g] = valid ? x[g] * scale : -INFINITY;
        need |= x[g] > m_run[g] + kRescaleThreshold;
      }
      // The producer may set sm_abort at any time, so whether to stop is decided
      // only by barrier reductions, whose result every consumer thread shares.
      const bool stop = !ok || *(volatile int*)&sm_abort != 0;
      if (tc::named_sync_or(1, 4 * 32, need || stop)) {
        // Rare: a wait gave up, or some head's maximum grew by more than 2^8.
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mx = warp_max(x[g]);
          if (lane == 0) wmax[warp * NP + g] = mx;
        }
        if (tc::named_sync_or(1, 4 * 32, stop)) {
          if (!ok) atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
          break;
        }
        float corr[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mt = fmaxf(fmaxf(wmax[g], wmax[NP + g]), fmaxf(wmax[2 * NP + g], wmax[3 * NP + g]));
          const float mn = fmaxf(m_run[g], mt);
          corr[g] = m_run[g] == -INFINITY ? 0.f : ex2(m_run[g] - mn);
          m_run[g] = mn;
          l_ex[g] *= corr[g];
          l_rd[g] *= corr[g];
        }
        if (kt > 0) {
          // O^T holds the earlier tiles (their P.V completed before S^T(kt) did).
          float o[16];
          tc::ld16(tmem + trow + kColO, o);
          tc::wait_ld();
#pragma unroll
          for (int g = 0; g < G; ++g) o[g] *= corr[g];
          tc::st16(tmem + trow + kColO, o);
          tc::wait_st();
        }
      }
      // P^T row of token tid (zero for padding heads and masked tokens).
      uint32_t pk[NP / 2], pl[NP / 2];
#pragma unroll
      for (int i = 0; i < NP / 2; ++i) {
        if (2 * i < G) {
          const float pa = ex2(x[2 * i] - m_run[2 * i]), pb = ex2(x[2 * i + 1] - m_run[2 * i + 1]);
          l_ex[2 * i] += pa;
          l_ex[2 * i + 1] += pb;
          pk[i] = pack2<T>(pa, pb);
          const float2 w = Elem<T>::to_f2(pk[i]);
          if constexpr (kBf16) {
            pl[i] = pack2<T>(pa - w.x, pb - w.y);
            const float2 z = Elem<T>::to_f2(pl[i]);
            l_rd[2 * i] += w.x + z.x;
            l_rd[2 * i + 1] += w.y + z.y;
          } else {
            pl[i] = 0u;
            l_rd[2 * i] += w.x;
            l_rd[2 * i + 1] += w.y;
          }
        } else {
          pk[i] = 0u;
          pl[i] = 0u;
        }
      }
      {
        const uint32_t roff = (tid >> 3) * 256 + (tid & 7) * 32;
        const int sw = (tid >> 2) & 1;  // 32-byte swizzle: 16-byte halves swap in rows 4..7
        uint8_t* prow = ps + roff;
        *reinterpret_cast<uint4*>(prow + (sw << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(prow + ((sw ^ 1) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        if constexpr (kBf16) {
          uint8_t* lrow = ps_lo + roff;
          *reinterpret_cast<uint4*>(lrow + (sw << 4)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          *reinterpret_cast<uint4*>(lrow + ((sw ^ 1) << 4)) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::named_sync(1, 4 * 32);
      if (tid == 0) {
        if (!issue_pv(kt)) {
          give_up();
          if (kt + 1 < ntiles) mbar_arrive(bar_s);
        } else if (kt + 1 < ntiles && !issue_s(kt + 1)) {
          give_up();
          mbar_arrive(bar_s);
        }
      }
      __syncwarp();
    }
    // Every MMA issued has completed once bar_o fires (commit with nothing pending
    // arrives at once).
    if (tid == 0) tc::commit(bar_o);
    __syncwarp();
    if (!mbar_wait(bar_o, 0)) {
      atomicOr(p.status, kStatusTimeout);
      *(volatile int*)&sm_abort = 1;
    }
    tc::fence_after_sync();
    float o[16];
    tc::ld16(tmem + trow + kColO, o);
    tc::wait_ld();
    // l and l~ over the 128 token rows: warp trees, then the four warps in order.
    float* red = wmax;  // [4 warps][2][16]
    tc::named_sync(1, 4 * 32);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float a = warp_sum(l_ex[g]), b = warp_sum(l_rd[g]);
      if (lane == 0) {
        red[warp * 2 * NP + g] = a;
        red[warp * 2 * NP + NP + g] = b;
      }
    }
    tc::fence_before_sync();
    __syncthreads();  // ring drained (the producer waited for its loads): reuse it
    if (*(volatile int*)&sm_abort == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) sm_acc[g * D + tid] = ntiles > 0 ? o[g] : 0.f;
      if (tid < G) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          a += red[w * 2 * NP + tid];
          b += red[w * 2 * NP + NP + tid];
        }
        float mrun = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) mrun = g == tid ? m_run[g] : mrun;
        sm_m[tid] = mrun;
        sm_l[tid] = a;
        sm_lr[tid] = b;
      }
    }
  } else if constexpr (PATH == kPathMmaKv8) {
    // ---------------- MMA consumers over an FP8 (E4M3) cache ----------------
    // Fragments are loaded straight from the 128-byte swizzled byte rows.  Two index
    // permutations make each thread's fragment bytes contiguous: the reduction index
    // of S = K q^T (k-step kk, thread quad t covers d = 16(2t + kk/4) + 4(kk%4) +
    // {0,1} for a0/a1/b0 and + {2,3} for a2/a3/b1, applied to K and to q alike), and
    // the rows of O^T (row g / g+8 of m-tile mi is dim 16g + 2mi / 16g + 2mi + 1,
    // undone when the state is written).  Widening is exact (cvt to f16).
    static_assert(D == 128, "FP8 K/V rows are single 128-byte swizzle rows");
    constexpr int KT = 8;                   // k-steps of S, m-tiles of O^T
    constexpr int NT = G >= 8 ? G / 8 : 1;  // N tiles of 8 query heads
    const int g = lane >> 2, t = lane & 3, qcol = 2 * t;
    uint32_t qb[NT][KT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int head = nt * 8 + g;
      const T* qh = reinterpret_cast<const T*>(p.q) +
                    ((int64_t)wk.b * p.Hq + wk.kvh * G + (head < G ? head : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const int dq = 16 * (2 * t + kk / 4) + 4 * (kk % 4);
        qb[nt][kk][0] = head < G ? *reinterpret_cast<const uint32_t*>(qh + dq) : 0u;
        qb[nt][kk][1] = head < G ? *reinterpret_cast<const uint32_t*>(qh + dq + 2) : 0u;
      }
    }
    float o[NT][KT][4];
    // l: sums of the fp32 weights (for lse); lr: of the 16-bit weights P.V uses (for out).
    float mA[NT], mB[NT], lA[NT], lB[NT], lrA[NT], lrB[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int mi = 0; mi < KT; ++mi) o[nt][mi][0] = o[nt][mi][1] = o[nt][mi][2] = o[nt][mi][3] = 0.f;
      mA[nt] = mB[nt] = -INFINITY;
      lA[nt] = lB[nt] = lrA[nt] = lrB[nt] = 0.f;
    }
    const float scale = p.scale_log2;
    // Each warp takes SUB groups of 16 tokens per tile: their K loads, widening and
    // score mma are independent chains, one max update covers all of them, and P.V
    // accumulates them into the same O^T fragments.
    constexpr int SUB = TILE / (kConsumerWarps * 16);
    static_assert(SUB * kConsumerWarps * 16 == TILE, "the FP8 tile splits into 16-token groups");
    const int tok0 = warp * 16 * SUB;

    for (int kt = 0; kt < ntiles; ++kt) {
      const int s = kt % NSLOT;
      const bool ok = mbar_wait(full_bar(s), (kt / NSLOT) & 1);
      if (__any_sync(0xffffffffu, !ok || *(volatile int*)&sm_abort != 0)) {
        if (!ok) {
          atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
        }
        break;
      }
      const int ntok = min(TILE, wk.t1 - (wk.t0 + kt * TILE));
      if (tok0 < ntok) {
        const uint8_t* kslot = smem + (size_t)s * kSlotBytes;
        const uint8_t* vslot = kslot + kRowsBytes;
        // Scores of every group: two accumulators each (even and odd k-steps) halve
        // the chains of dependent mma.
        float sc[SUB][NT][4];
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
          const int tb = tok0 + 16 * u;
          // K: rows tb + g (+8), 16-byte chunks 2t and 2t + 1.
          uint4 kw[2][2];
#pragma unroll
          for (int rh = 0; rh < 2; ++rh)
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
              const int r = tb + g + 8 * rh, c = 2 * t + grp;
              kw[rh][grp] = *reinterpret_cast<const uint4*>(kslot + r * 128 + ((c ^ (r & 7)) << 4));
            }
          float sd[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[u][nt][i] = sd[nt][i] = 0.f;
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            const uint4& w0 = kw[0][kk >> 2];
            const uint4& w1 = kw[1][kk >> 2];
            const int wi = kk & 3;
            const uint32_t x0 = wi == 0 ? w0.x : wi == 1 ? w0.y : wi == 2 ? w0.z : w0.w;
            const uint32_t x1 = wi == 0 ? w1.x : wi == 1 ? w1.y : wi == 2 ? w1.z : w1.w;
            uint32_t a[4];
            e4m3x4_to_f16x4(x0, a[0], a[2]);  // bytes 0, 1 and 2, 3 of row g
            e4m3x4_to_f16x4(x1, a[1], a[3]);  // the same of row g + 8
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<T>((kk & 1) ? sd[nt] : sc[u][nt], a, qb[nt][kk][0], qb[nt][kk][1]);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[u][nt][i] += sd[nt][i];
        }
        uint32_t pb0[SUB][NT], pb1[SUB][NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sA0[SUB], sB0[SUB], sA1[SUB], sB1[SUB];
          float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
          for (int u = 0; u < SUB; ++u) {
            const bool v0 = tok0 + 16 * u + g < ntok, v1 = tok0 + 16 * u + g + 8 < ntok;
            sA0[u] = v0 ? sc[u][nt][0] * scale : -INFINITY;
            sB0[u] = v0 ? sc[u][nt][1] * scale : -INFINITY;
            sA1[u] = v1 ? sc[u][nt][2] * scale : -INFINITY;
            sB1[u] = v1 ? sc[u][nt][3] * scale : -INFINITY;
            xA = fmaxf(xA, fmaxf(sA0[u], sA1[u]));
            xB = fmaxf(xB, fmaxf(sB0[u], sB1[u]));
          }
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, off));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, off));
          }
          if (xA > mA[nt] + kRescaleThreshold) {
            const float corr = ex2(mA[nt] - xA);
            lA[nt] *= corr;
            lrA[nt] *= corr;
#pragma unroll
            for (int mi = 0; mi < KT; ++mi) { o[nt][mi][0] *= corr; o[nt][mi][2] *= corr; }
            mA[nt] = xA;
          }
          if (xB > mB[nt] + kRescaleThreshold) {
            const float corr = ex2(mB[nt] - xB);
            lB[nt] *= corr;
            lrB[nt] *= corr;
#pragma unroll
            for (int mi = 0; mi < KT; ++mi) { o[nt][mi][1] *= corr; o[nt][mi][3] *= corr; }
            mB[nt] = xB;
          }
          // Row tok0 is valid, so the column maxima (and mA, mB) are finite here.
#pragma unroll
          for (int u = 0; u < SUB; ++u) {
            const float pA0 = ex2(sA0[u] - mA[nt]), pB0 = ex2(sB0[u] - mB[nt]);
            const float pA1 = ex2(sA1[u] - mA[nt]), pB1 = ex2(sB1[u] - mB[nt]);
            lA[nt] += pA0 + pA1;
            lB[nt] += pB0 + pB1;
            const uint32_t r0 = pack2<T>(pA0, pB0), r1 = pack2<T>(pA1, pB1);
            // lr sums the same 16-bit weights that P.V multiplies, so the output is an
            // exact convex combination of V rows under the rounded weights.
            const float2 w0 = Elem<T>::to_f2(r0), w1 = Elem<T>::to_f2(r1);
            lrA[nt] += w0.x + w1.x;
            lrB[nt] += w0.y + w1.y;
            pb0[u][nt] = movmatrix_trans(r0);
            pb1[u][nt] = movmatrix_trans(r1);
          }
        }
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
          const int tb = tok0 + 16 * u;
          // V^T: token rows tb + 2t, +1, +8, +9; the 16-byte chunk g (dims 16g ..).
          uint4 vw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = tb + 2 * t + (i & 1) + 8 * (i >> 1);
            vw[i] = *reinterpret_cast<const uint4*>(vslot + r * 128 + ((g ^ (r & 7)) << 4));
          }
#pragma unroll
          for (int mi = 0; mi < KT; ++mi) {
            const int wi = mi >> 1;
            const uint32_t k = 2u * (mi & 1);
            const uint32_t y0 = wi == 0 ? vw[0].x : wi == 1 ? vw[0].y : wi == 2 ? vw[0].z : vw[0].w;
            const uint32_t y1 = wi == 0 ? vw[1].x : wi == 1 ? vw[1].y : wi == 2 ? vw[1].z : vw[1].w;
            const uint32_t y2 = wi == 0 ? vw[2].x : wi == 1 ? vw[2].y : wi == 2 ? vw[2].z : vw[2].w;
            const uint32_t y3 = wi == 0 ? vw[3].x : wi == 1 ? vw[3].y : wi == 2 ? vw[3].z : vw[3].w;
            // bytes k (dim 16g + 2mi) and k + 1 (dim 16g + 2mi + 1) of two token rows,
            // gathered as [row0 k, row1 k, row0 k+1, row1 k+1]: each widened pair holds
            // the row of the first word in its low half, the second in its high half
            const uint32_t sel = ((5u + k) << 12) | ((1u + k) << 8) | ((4u + k) << 4) | k;
            uint32_t a[4], z;
            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(z) : "r"(y0), "r"(y1), "r"(sel));
            e4m3x4_to_f16x4(z, a[0], a[1]);
            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(z) : "r"(y2), "r"(y3), "r"(sel));
            e4m3x4_to_f16x4(z, a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816<T>(o[nt][mi], a, pb0[u][nt], pb1[u][nt]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        lA[nt] += __shfl_xor_sync(0xffffffffu, lA[nt], off);
        lB[nt] += __shfl_xor_sync(0xffffffffu, lB[nt], off);
        lrA[nt] += __shfl_xor_sync(0xffffffffu, lrA[nt], off);
        lrB[nt] += __shfl_xor_sync(0xffffffffu, lrB[nt], off);
      }
    }
    __syncthreads();  // ring drained: reuse it for the per-warp states
    if (*(volatile int*)&sm_abort == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int hA = nt * 8 + qcol;
        if (hA < G) {
          float* accA = sm_acc + (warp * G + hA) * D;
          float* accB = accA + D;
#pragma unroll
          for (int mi = 0; mi < KT; ++mi) {
            accA[16 * g + 2 * mi] = o[nt][mi][0];
            accB[16 * g + 2 * mi] = o[nt][mi][1];
            accA[16 * g + 2 * mi + 1] = o[nt][mi][2];
            accB[16 * g + 2 * mi + 1] = o[nt][mi][3];
          }
          if (g == 0) {
            sm_m[warp * G + hA] = mA[nt];
            sm_m[warp * G + hA + 1] = mB[nt];
            sm_l[warp * G + hA] = lA[nt];
            sm_l[warp * G + hA + 1] = lB[nt];
            sm_lr[warp * G + hA] = lrA[nt];
            sm_lr[warp * G + hA + 1] = lrB[nt];
          }
        }
      }
    }
  } else if constexpr (PATH == kPathMma) {
    // ---------------- MMA consumers ----------------
    constexpr int KT = D / 16;            // k-steps of S = K Q^T, m-tiles of O^T
    constexpr int NT = G >= 8 ? G / 8 : 1;  // N tiles of 8 query heads
    const int qrow = lane >> 2;           // C/B fragment row (token) or column (head)
    const int qcol = (lane & 3) * 2;      // C fragment column pair (heads qcol, qcol+1)
    const int mj = lane >> 3, mr = lane & 7;  // ldmatrix: matrix and row this lane addresses
    // q as the B operand of S^T = K Q^T: B[k][n] = q[head n][k]; heads >= G are zero.
    uint32_t qb[NT][KT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int head = nt * 8 + qrow;
      const T* qh = reinterpret_cast<const T*>(p.q) +
                    ((int64_t)wk.b * p.Hq + wk.kvh * G + (head < G ? head : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        qb[nt][kk][0] = head < G ? *reinterpret_cast<const uint32_t*>(qh + kk * 16 + qcol) : 0u;
        qb[nt][kk][1] = head < G ? *reinterpret_cast<const uint32_t*>(qh + kk * 16 + qcol + 8) : 0u;
      }
    }
    float o[NT][KT][4];
    // l: sums of the fp32 weights (for lse); lr: of the 16-bit weights P.V uses (for out).
    float mA[NT], mB[NT], lA[NT], lB[NT], lrA[NT], lrB[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int mi = 0; mi < KT; ++mi) o[nt][mi][0] = o[nt][mi][1] = o[nt][mi][2] = o[nt][mi][3] = 0.f;
      mA[nt] = mB[nt] = -INFINITY;
      lA[nt] = lB[nt] = lrA[nt] = lrB[nt] = 0.f;
    }
    const float scale = p.scale_log2;
    // bf16 weights carry 8 significant bits: a weight rounded once is off by up to
    // 2^-9 of itself, which over a few tokens moves out by more than the tolerance.
    // So P.V takes each bf16 weight as hi + lo (two bf16 values, 16 significant bits
    // together) in two mma; f16 (11 bits) needs no split.
    constexpr bool kSplitP = Elem<T>::kMantissaBits < 11;
    const int tok0 = warp * 16;
    const int krow = tok0 + (mj & 1) * 8 + mr;   // K rows this lane addresses (A = K)
    const int vrow = tok0 + (mj >> 1) * 8 + mr;  // V rows this lane addresses (A = V^T)

    for (int kt = 0; kt < ntiles; ++kt) {
      const int s = kt % NSLOT;
      const bool ok = mbar_wait(full_bar(s), (kt / NSLOT) & 1);
      if (__any_sync(0xffffffffu, !ok || *(volatile int*)&sm_abort != 0)) {
        if (!ok) {
          atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
        }
        break;
      }
      const int ntok = min(TILE, wk.t1 - (wk.t0 + kt * TILE));
      if (tok0 < ntok) {
        const uint32_t kbase = smem_addr(smem + (size_t)s * kSlotBytes);
        const uint32_t vbase = kbase + kRowsBytes;
        // Two accumulators (even and odd k-steps) halve the chain of dependent mma.
        float sc[NT][4], sd[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[nt][i] = sd[nt][i] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          uint32_t a[4];
          ldmatrix_x4(a, swz_addr(kbase, TILE, krow, 2 * kk + (mj >> 1)));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma16816<T>((kk & 1) ? sd[nt] : sc[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[nt][i] += sd[nt][i];
        const bool v0 = tok0 + qrow < ntok, v1 = tok0 + qrow + 8 < ntok;
        uint32_t pb0[NT], pb1[NT], pc0[NT], pc1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float sA0 = v0 ? sc[nt][0] * scale : -INFINITY;
          const float sB0 = v0 ? sc[nt][1] * scale : -INFINITY;
          const float sA1 = v1 ? sc[nt][2] * scale : -INFINITY;
          const float sB1 = v1 ? sc[nt][3] * scale : -INFINITY;
          float xA = fmaxf(sA0, sA1), xB = fmaxf(sB0, sB1);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, off));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, off));
          }
          if (xA > mA[nt] + kRescaleThreshold) {
            const float corr = ex2(mA[nt] - xA);
            lA[nt] *= corr;
            lrA[nt] *= corr;
#pragma unroll
            for (int mi = 0; mi < KT; ++mi) { o[nt][mi][0] *= corr; o[nt][mi][2] *= corr; }
            mA[nt] = xA;
          }
          if (xB > mB[nt] + kRescaleThreshold) {
            const float corr = ex2(mB[nt] - xB);
            lB[nt] *= corr;
            lrB[nt] *= corr;
#pragma unroll
            for (int mi = 0; mi < KT; ++mi) { o[nt][mi][1] *= corr; o[nt][mi][3] *= corr; }
            mB[nt] = xB;
          }
          // Row tok0 is valid, so the column maxima (and mA, mB) are finite here.
          const float pA0 = ex2(sA0 - mA[nt]), pB0 = ex2(sB0 - mB[nt]);
          const float pA1 = ex2(sA1 - mA[nt]), pB1 = ex2(sB1 - mB[nt]);
          lA[nt] += pA0 + pA1;
          lB[nt] += pB0 + pB1;
          const uint32_t r0 = pack2<T>(pA0, pB0), r1 = pack2<T>(pA1, pB1);
          // lr sums the same 16-bit weights that P.V multiplies (numerator and
          // normaliser of out see one set of weights).
          const float2 w0 = Elem<T>::to_f2(r0), w1 = Elem<T>::to_f2(r1);
          if constexpr (kSplitP) {
            const uint32_t t0 = pack2<T>(pA0 - w0.x, pB0 - w0.y), t1 = pack2<T>(pA1 - w1.x, pB1 - w1.y);
            const float2 z0 = Elem<T>::to_f2(t0), z1 = Elem<T>::to_f2(t1);
            lrA[nt] += (w0.x + z0.x) + (w1.x + z1.x);
            lrB[nt] += (w0.y + z0.y) + (w1.y + z1.y);
            pc0[nt] = movmatrix_trans(t0);
            pc1[nt] = movmatrix_trans(t1);
          } else {
            lrA[nt] += w0.x + w1.x;
            lrB[nt] += w0.y + w1.y;
          }
          // P (tokens x heads, accumulator layout) -> P^T as the B operand (k = token).
          pb0[nt] = movmatrix_trans(r0);
          pb1[nt] = movmatrix_trans(r1);
        }
#pragma unroll
        for (int mi = 0; mi < KT; ++mi) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, swz_addr(vbase, TILE, vrow, 2 * mi + (mj & 1)));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816<T>(o[nt][mi], a, pb0[nt], pb1[nt]);
            if constexpr (kSplitP) mma16816<T>(o[nt][mi], a, pc0[nt], pc1[nt]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
    // Row sums: lanes sharing a head pair hold partial sums over their tokens.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        lA[nt] += __shfl_xor_sync(0xffffffffu, lA[nt], off);
        lB[nt] += __shfl_xor_sync(0xffffffffu, lB[nt], off);
        lrA[nt] += __shfl_xor_sync(0xffffffffu, lrA[nt], off);
        lrB[nt] += __shfl_xor_sync(0xffffffffu, lrB[nt], off);
      }
    }
    __syncthreads();  // ring drained: reuse it for the per-warp states
    if (*(volatile int*)&sm_abort == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int hA = nt * 8 + qcol;
        if (hA < G) {
          float* accA = sm_acc + (warp * G + hA) * D;
          float* accB = accA + D;
#pragma unroll
          for (int mi = 0; mi < KT; ++mi) {
            accA[16 * mi + qrow] = o[nt][mi][0];
            accB[16 * mi + qrow] = o[nt][mi][1];
            accA[16 * mi + qrow + 8] = o[nt][mi][2];
            accB[16 * mi + qrow + 8] = o[nt][mi][3];
          }
          if (qrow == 0) {
            sm_m[warp * G + hA] = mA[nt];
            sm_m[warp * G + hA + 1] = mB[nt];
            sm_l[warp * G + hA] = lA[nt];
            sm_l[warp * G + hA + 1] = lB[nt];
            sm_lr[warp * G + hA] = lrA[nt];
            sm_lr[warp * G + hA + 1] = lrB[nt];
          }
        }
      }
    }
  } else {
    // ---------------- FFMA consumers ----------------
    constexpr int LPT = (G * D > 512) ? 16 : 8;  // lanes per token
    constexpr int DL = D / LPT;                   // dimensions per lane
    constexpr int NCH = DL / 8;                   // 16-byte chunks per lane per row
    constexpr int GPW = 32 / LPT;                 // token groups per warp
    constexpr int TPG = TILE / NGRP;              // tokens per group per stage
    static_assert(TILE % NGRP == 0, "tile must split evenly over token groups");
    const int j = lane % LPT;                     // lane within its token group
    const int gi = warp * GPW + lane / LPT;       // token group id
    float acc[G][DL];
    float m_run[G], l_run[G];
    const T* qg = reinterpret_cast<const T*>(p.q) + ((int64_t)wk.b * p.Hq + wk.kvh * G) * D;
    float qf[G][DL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(qg + g * D + (j + LPT * c) * 8);
        unpack8<T>(raw, &qf[g][c * 8]);
      }
#pragma unroll
      for (int e = 0; e < DL; ++e) qf[g][e] *= p.scale_log2;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[g][e] = 0.f;
    }

    for (int kt = 0; kt < ntiles; ++kt) {
      const int s = kt % NSLOT;
      // Every lane waits; the warp leaves together so shuffles never see a partial warp.
      const bool ok = mbar_wait(full_bar(s), (kt / NSLOT) & 1);
      if (__any_sync(0xffffffffu, !ok || *(volatile int*)&sm_abort != 0)) {
        if (!ok) {
          atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
        }
        break;
      }
      const int ntok = min(TILE, wk.t1 - (wk.t0 + kt * TILE));
      const T* Ks = reinterpret_cast<const T*>(smem + (size_t)s * kSlotBytes);
      const T* Vs = Ks + TILE * D;

      float sc[TPG][G];
#pragma unroll
      for (int r = 0; r < TPG; ++r) {
        const int tok = gi + NGRP * r;
        float part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = 0.f;
        if (tok < ntok) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const uint4 raw = *reinterpret_cast<const uint4*>(Ks + tok * D + (j + LPT * c) * 8);
            float kf[8];
            unpack8<T>(raw, kf);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int e = 0; e < 8; ++e) part[g] = fmaf(qf[g][c * 8 + e], kf[e], part[g]);
          }
        }
#pragma unroll
        for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) part[g] += __shfl_xor_sync(0xffffffffu, part[g], off);
#pragma unroll
        for (int g = 0; g < G; ++g) sc[r][g] = (tok < ntok) ? part[g] : -INFINITY;
      }

      float pr[TPG][G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = sc[0][g];
#pragma unroll
        for (int r = 1; r < TPG; ++r) mx = fmaxf(mx, sc[r][g]);
        if (mx > m_run[g] + kRescaleThreshold) {
          const float corr = ex2(m_run[g] - mx);
          l_run[g] *= corr;
#pragma unroll
          for (int e = 0; e < DL; ++e) acc[g][e] *= corr;
          m_run[g] = mx;
        }
#pragma unroll
        for (int r = 0; r < TPG; ++r) {
          pr[r][g] = (gi + NGRP * r < ntok) ? ex2(sc[r][g] - m_run[g]) : 0.f;
          l_run[g] += pr[r][g];
        }
      }

#pragma unroll
      for (int r = 0; r < TPG; ++r) {
        const int tok = gi + NGRP * r;
        if (tok < ntok) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const uint4 raw = *reinterpret_cast<const uint4*>(Vs + tok * D + (j + LPT * c) * 8);
            float vf[8];
            unpack8<T>(raw, vf);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[g][c * 8 + e] = fmaf(pr[r][g], vf[e], acc[g][c * 8 + e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
    __syncthreads();  // ring drained: reuse it for the per-group states
    if (*(volatile int*)&sm_abort == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float4* dst = reinterpret_cast<float4*>(sm_acc + (gi * G + g) * D + (j + LPT * c) * 8);
          dst[0] = make_float4(acc[g][c * 8 + 0], acc[g][c * 8 + 1], acc[g][c * 8 + 2], acc[g][c * 8 + 3]);
          dst[1] = make_float4(acc[g][c * 8 + 4], acc[g][c * 8 + 5], acc[g][c * 8 + 6], acc[g][c * 8 + 7]);
        }
      if (j == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          sm_m[gi * G + g] = m_run[g];
          sm_l[gi * G + g] = l_run[g];
          sm_lr[gi * G + g] = l_run[g];  // fp32 weights: P.V used the same ones
        }
      }
    }
  }
  __syncthreads();
  if constexpr (PATH == kPathUmma) {
    if (warp == 0) {  // the allocating warp; every tensor-memory read has completed
      tc::fence_after_sync();
      tc::tmem_dealloc(*tmem_slot, kTmemCols);
    }
  }
  // A CTA whose pipeline gave up (the status word says so) still finishes, with an
  // empty partial: its (sequence, KV head) counter must complete and return to zero,
  // and a CTA of a cluster must still reach the cluster barriers.
  finish_cta<T, D, G, NGRP, kMode, kSeg, kPair>(p, wk, sm_acc, sm_last, sm_abort != 0, smem, kRing,
                                         combine_bars);
}

// Two-launch ablation, second kernel: one CTA per (sequence, KV head) combines
// the partials written by fd_split_kernel<..., MODE = 1>.
template <typename T, int D, int G, int PATH>
__global__ void __launch_bounds__(kThreads, 2) fd_combine_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;  // bulk copies need 16-byte alignment only
  constexpr uint32_t kBytes = (uint32_t)ring_bytes_for(PATH, D, 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBytes);  // kCombineBars of them
  static_assert(kCombineBars * 8 <= kRingMetaBytes, "combine barriers fit after the ring");
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int j = 0; j < kCombineBars; ++j) mbar_init(smem_addr(bars + j), 1);
    fence_mbar_init();
  }
  pdl_wait();
  __syncthreads();
  const int b = blockIdx.x / p.Hkv, kvh = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
  uint32_t phase = 0;
  combine_partials<T, D, G>(p, b, kvh, p.wseg[b] * p.rps, rec_base(p, b), 0, G, smem, kBytes,
                            smem_addr(bars), phase);
}

}  // namespace dev

template <typename T, int D, int G, int PATH>
cudaError_t launch_dgp(const Params& p, int mode, bool pdl, int grid, cudaStream_t stream) {
  // The shallow-ring build exists for the fused mma.sync kernel with G <= 8 only (the
  // planner asks for it nowhere else; at G = 16 it would not fit its registers).
  constexpr bool kHasShallow = PATH == kPathMma && G <= 8;
  const bool shallow = kHasShallow && mode == 0 && p.ctas_per_sm == kShallowCtasPerSm;
  const size_t smem = smem_bytes_for(PATH, D, shallow ? kShallowCtasPerSm : 2);
  // The split kernels of plans that merge segments in clusters are separate
  // instantiations (kernel modes 4 and 5).
  // Mode 6 (every partial of a pair in one cluster) comes from the host; the split
  // kernels of plans that merge segments in clusters are kernel modes 4 and 5.
  const bool seg = mode <= 1 && p.rps != p.C;
  const int kmode = seg ? mode + 4 : shallow ? 7 : mode;
  const void* fn;
  switch (kmode) {
    case 0: fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, PATH, 0>); break;
    case 7:
      fn = reinterpret_cast<const void*>(
          &dev::fd_split_kernel<T, D, G, PATH, 0, kHasShallow ? kShallowCtasPerSm : 2>);
      break;
    case 1: fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, PATH, 1>); break;
    case 2: fn = reinterpret_cast<const void*>(&dev::fd_combine_kernel<T, D, G, PATH>); break;
    case 3: fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, PATH, 3>); break;
    case 4: fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, PATH, 4>); break;
    case 5: fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, PATH, 5>); break;
    default: fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, PATH, 6>); break;
  }
  int dev_id = 0;
  cudaError_t err = cudaGetDevice(&dev_id);
  if (err != cudaSuccess) return err;
  // The opt-in shared-memory size (and, for clusters of more than 8 CTAs, the
  // non-portable cluster size) are per-device function attributes.
  static uint64_t done_mask[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint64_t bit = 1ull << (dev_id & 63);
  if (!(__atomic_load_n(&done_mask[kmode], __ATOMIC_ACQUIRE) & bit)) {
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err == cudaSuccess && kmode == 6)
      err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    __atomic_fetch_or(&done_mask[kmode], bit, __ATOMIC_RELEASE);
  }
  void* args[] = {const_cast<Params*>(&p)};
  cudaLaunchAttribute attr[2];
  unsigned int nattr = 1;
  if (mode == 3) {
    // The designated combiners wait for other CTAs: the whole grid must be resident.
    int per_sm = 0, sms = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev_id);
    if (err != cudaSuccess) return err;
    if ((int64_t)per_sm * sms < grid) return cudaErrorCooperativeLaunchTooLarge;
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    if (seg || kmode == 6) {
      // The C chunk CTAs of a segment, or all W C partial CTAs of a (sequence, KV
      // head) pair (consecutive block indices), form one cluster.
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = (unsigned)(kmode == 6 ? p.pair_cluster : p.C);
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      nattr = 2;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Launchers per consumer family, each instantiated in its own translation unit
// (parallel builds): CUDA-core consumers, and mma.sync consumers (16-bit and E4M3).
template <typename T>
cudaError_t launch_typed_ffma(const Params& p, int d, int G, int mode, bool pdl, int grid,
                              cudaStream_t s) {
#define FD_CASE(DD, GG) \
  if (d == DD && G == GG) return launch_dgp<T, DD, GG, kPathFfma>(p, mode, pdl, grid, s);
  FD_CASE(64, 1) FD_CASE(64, 2) FD_CASE(64, 4) FD_CASE(64, 8)
  FD_CASE(128, 1) FD_CASE(128, 2) FD_CASE(128, 4) FD_CASE(128, 8)
#undef FD_CASE
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_typed_mma(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                             cudaStream_t s) {
#define FD_CASE(DD, GG, PP) \
  if (d == DD && G == GG && path == PP) return launch_dgp<T, DD, GG, PP>(p, mode, pdl, grid, s);
  FD_CASE(64, 4, kPathMma) FD_CASE(64, 8, kPathMma) FD_CASE(64, 16, kPathMma)
  FD_CASE(128, 4, kPathMma) FD_CASE(128, 8, kPathMma) FD_CASE(128, 16, kPathMma)
  if constexpr (std::is_same<T, __half>::value) {
    FD_CASE(128, 4, kPathMmaKv8) FD_CASE(128, 8, kPathMmaKv8) FD_CASE(128, 16, kPathMmaKv8)
  }
#undef FD_CASE
  return cudaErrorInvalidValue;
}

// The tcgen05 consumers (d = 128, G in {4, 8, 16}); their own translation units.
template <typename T>
cudaError_t launch_typed_umma(const Params& p, int d, int G, int mode, bool pdl, int grid,
                              cudaStream_t s) {
  if (d == 128 && G == 4) return launch_dgp<T, 128, 4, kPathUmma>(p, mode, pdl, grid, s);
  if (d == 128 && G == 8) return launch_dgp<T, 128, 8, kPathUmma>(p, mode, pdl, grid, s);
  if (d == 128 && G == 16) return launch_dgp<T, 128, 16, kPathUmma>(p, mode, pdl, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace fd
