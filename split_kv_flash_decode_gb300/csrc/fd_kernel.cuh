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
//   * warp 4, lane 0: TMA producer.  Per stage it issues two 3-D tensor loads
//     (kTile K rows and kTile V rows of one KV head) into an mbarrier ring.
//   * warps 0-3: consumers.  Lanes form groups of LPT lanes; a group owns one
//     token at a time, each lane holding D/LPT dimensions of q (fp32, scaled into
//     the log2 domain) for all G query heads that share this KV head, so every
//     K/V byte loaded serves the whole GQA group.  Scores use FFMA plus an
//     xor-shuffle reduction inside the group; each group keeps its own running
//     (m, l, acc) with a lazy rescale (only when the max grows by > 2^8).
//   * end of CTA: groups merge through shared memory into one fp32 partial,
//     which is written to the workspace; one thread then does
//     fence + atom.add.acq_rel.gpu on the (sequence, KV head) arrival counter.
//     The CTA that sees count == Wtot - 1 is the last arriver: it combines the
//     Wtot partials in index order (deterministic), writes out and lse, and
//     resets the counter.  No CTA ever waits for another, so the kernel cannot
//     deadlock; the only waits are bounded mbarrier waits on its own loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fd_common.h"

namespace fd {
namespace dev {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr float kLn2 = 0.693147180559945309417f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits give up after ~1 s

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

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 3-D tiled TMA load: box at coordinates (c0, c1, c2) of `map` into shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
struct Elem;

template <>
struct Elem<__half> {
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return __half22float2(h);
  }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

template <>
struct Elem<__nv_bfloat16> {
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

// Work item of CTA `cta` in the flattened (sequence, slot, KV head) order.
struct Work {
  int b, kvh, slot, wtot, t0, t1;
  int64_t pbase;  // index of the first partial of sequence b
};

__device__ __forceinline__ Work decode_work(const Params& p, int cta) {
  int lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.unit_base[mid] <= cta) lo = mid; else hi = mid;
  }
  Work w;
  w.b = lo;
  const int r = cta - p.unit_base[lo];
  w.kvh = r % p.Hkv;
  w.slot = r / p.Hkv;
  w.wtot = (p.unit_base[lo + 1] - p.unit_base[lo]) / p.Hkv;
  const int L = p.cu[lo + 1] - p.cu[lo];
  chunk_range(L, p.wseg[lo], p.C, w.slot, &w.t0, &w.t1);
  w.pbase = (int64_t)(p.unit_base[lo] / p.Hkv) * p.Hq;
  return w;
}

// OnlineSoftmaxCombine of the Wtot partials of (b, kvh): all kThreads threads take
// part; `sm` holds at least G * wtot + 2 * G floats.  Order of summation is fixed
// (partial index order), so the result does not depend on arrival order.
template <typename T, int D, int G>
__device__ __forceinline__ void combine_partials(const Params& p, int b, int kvh, int wtot,
                                                 int64_t pbase, float* sm) {
  float* coef = sm;              // [G][wtot]  e^{m_w - M}
  float* ML = sm + G * wtot;     // [G][2]     (M, Lambda)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kThreads / 32;
  for (int g = warp; g < G; g += kWarps) {
    const int64_t row = pbase + (int64_t)(kvh * G + g) * wtot;
    float M = -INFINITY;
    for (int w = lane; w < wtot; w += 32) M = fmaxf(M, __ldcg(p.part_m + row + w));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float lam = 0.f;
    for (int w = lane; w < wtot; w += 32) {
      const float e = (M == -INFINITY) ? 0.f : ex2(__ldcg(p.part_m + row + w) - M);
      coef[g * wtot + w] = e;
      lam = fmaf(e, __ldcg(p.part_l + row + w), lam);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
    if (lane == 0) {
      ML[2 * g] = M;
      ML[2 * g + 1] = lam;
    }
  }
  __syncthreads();
  T* out = reinterpret_cast<T*>(p.out);
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, dim = idx - (idx / D) * D;
    const float* po = p.part_o + (pbase + (int64_t)(kvh * G + g) * wtot) * D + dim;
    const float* cg = coef + g * wtot;
    float a = 0.f;
    int w = 0;
    for (; w + 8 <= wtot; w += 8) {
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = __ldcg(po + (int64_t)(w + u) * D);
#pragma unroll
      for (int u = 0; u < 8; ++u) a = fmaf(cg[w + u], x[u], a);
    }
    for (; w < wtot; ++w) a = fmaf(cg[w], __ldcg(po + (int64_t)w * D), a);
    const float lam = ML[2 * g + 1];
    out[((int64_t)b * p.Hq + kvh * G + g) * D + dim] = Elem<T>::from_f(lam > 0.f ? a / lam : 0.f);
  }
  if (tid < G && p.lse != nullptr) {
    const float M = ML[2 * tid], lam = ML[2 * tid + 1];
    p.lse[(int64_t)b * p.Hq + kvh * G + tid] = lam > 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
  }
}

// MODE 0: fused split + last-arriver combine.  MODE 1: split only (partials).
template <typename T, int D, int G, int MODE>
__global__ void __launch_bounds__(kThreads, 2) fd_split_kernel(const __grid_constant__ Params p) {
  constexpr int STAGES = stages_for(D);
  constexpr int LPT = (G * D > 512) ? 16 : 8;  // lanes per token
  constexpr int DL = D / LPT;                   // dimensions per lane
  constexpr int NCH = DL / 8;                   // 16-byte chunks per lane per row
  constexpr int GPW = 32 / LPT;                 // token groups per warp
  constexpr int NGRP = kConsumerWarps * GPW;    // token groups per CTA
  constexpr int TPG = kTile / NGRP;             // tokens per group per stage
  constexpr uint32_t kRowsBytes = kTile * D * sizeof(T);
  static_assert(kTile % NGRP == 0, "tile must split evenly over token groups");
  static_assert(NGRP * G * D * 4 + 4 * NGRP * G * 4 <= STAGES * 2 * kRowsBytes,
                "group merge must fit in the ring");

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)STAGES * 2 * kRowsBytes);
  int& sm_abort = *reinterpret_cast<int*>(bars + 2 * STAGES);
  int& sm_last = *(reinterpret_cast<int*>(bars + 2 * STAGES) + 1);
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + STAGES + s); };
  auto k_rows = [&](int s) { return reinterpret_cast<const T*>(smem + (size_t)s * 2 * kRowsBytes); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Work wk = decode_work(p, blockIdx.x);
  const int ntiles = (wk.t1 - wk.t0 + kTile - 1) / kTile;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumerWarps);
    }
    fence_mbar_init();
    sm_abort = 0;
  }
  __syncthreads();

  // Per-group online-softmax state (consumers only).
  float acc[G][DL];
  float m_run[G], l_run[G];
  const int j = lane % LPT;                     // lane within its token group
  const int gi = warp * GPW + lane / LPT;       // token group id

  if (warp == kConsumerWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && ntiles > 0) {
      const uint64_t policy = l2_evict_first_policy();
      const int row0 = p.cu[wk.b] + wk.t0;
      int kt = 0;
      for (; kt < ntiles; ++kt) {
        const int s = kt % STAGES;
        if (kt >= STAGES && !mbar_wait(empty_bar(s), ((kt / STAGES) - 1) & 1)) {
          atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
          break;
        }
        if (*(volatile int*)&sm_abort) break;
        const uint32_t dst = smem_addr(smem + (size_t)s * 2 * kRowsBytes);
        mbar_arrive_expect_tx(full_bar(s), 2 * kRowsBytes);
        tma_load_3d(dst, &p.tm_k, 0, wk.kvh, row0 + kt * kTile, full_bar(s), policy);
        tma_load_3d(dst + kRowsBytes, &p.tm_v, 0, wk.kvh, row0 + kt * kTile, full_bar(s), policy);
      }
      // Every load issued must land before shared memory is reused or released.
      for (int t = (kt > STAGES ? kt - STAGES : 0); t < kt; ++t) {
        if (!mbar_wait(full_bar(t % STAGES), (t / STAGES) & 1)) atomicOr(p.status, kStatusTimeout);
      }
    }
  } else {
    // ---------------- consumers ----------------
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
      const int s = kt % STAGES;
      // Every lane waits; the warp leaves together so shuffles never see a partial warp.
      const bool ok = mbar_wait(full_bar(s), (kt / STAGES) & 1);
      if (__any_sync(0xffffffffu, !ok || *(volatile int*)&sm_abort != 0)) {
        if (!ok) {
          atomicOr(p.status, kStatusTimeout);
          *(volatile int*)&sm_abort = 1;
        }
        break;
      }
      const int ntok = min(kTile, wk.t1 - (wk.t0 + kt * kTile));
      const T* Ks = k_rows(s);
      const T* Vs = Ks + kTile * D;

      // Scores of this group's tokens for all G heads (log2 domain).
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

      // Online softmax with lazy rescaling.
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

      // P . V
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
  }
  __syncthreads();
  if (sm_abort) return;

  // ---------------- merge the token groups into one partial ----------------
  float* sm_acc = reinterpret_cast<float*>(smem);  // [NGRP][G][D]
  float* sm_m = sm_acc + NGRP * G * D;              // [NGRP][G]
  float* sm_l = sm_m + NGRP * G;                    // [NGRP][G]
  float* sm_fac = sm_l + NGRP * G;                  // [NGRP][G]
  float* sm_ML = sm_fac + NGRP * G;                 // [G][2]
  if (warp < kConsumerWarps) {
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
      }
    }
  }
  __syncthreads();
  if (tid < G) {
    const int g = tid;
    float M = -INFINITY;
    for (int q = 0; q < NGRP; ++q) M = fmaxf(M, sm_m[q * G + g]);
    float lam = 0.f;
    for (int q = 0; q < NGRP; ++q) {
      const float f = (M == -INFINITY) ? 0.f : ex2(sm_m[q * G + g] - M);
      sm_fac[q * G + g] = f;
      lam = fmaf(sm_l[q * G + g], f, lam);
    }
    sm_ML[2 * g] = M;
    sm_ML[2 * g + 1] = lam;
  }
  __syncthreads();

  const int h0 = wk.kvh * G;
  if (MODE == 0 && wk.wtot == 1) {
    // A single partial is already the answer: normalise and store.
    T* out = reinterpret_cast<T*>(p.out);
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int g = idx / D, dim = idx - (idx / D) * D;
      float a = 0.f;
#pragma unroll 4
      for (int q = 0; q < NGRP; ++q) a = fmaf(sm_acc[(q * G + g) * D + dim], sm_fac[q * G + g], a);
      const float lam = sm_ML[2 * g + 1];
      out[((int64_t)wk.b * p.Hq + h0 + g) * D + dim] = Elem<T>::from_f(lam > 0.f ? a / lam : 0.f);
    }
    if (tid < G && p.lse != nullptr) {
      const float M = sm_ML[2 * tid], lam = sm_ML[2 * tid + 1];
      p.lse[(int64_t)wk.b * p.Hq + h0 + tid] = lam > 0.f ? (M + log2f(lam)) * kLn2 : -INFINITY;
    }
    return;
  }

  // Publish this CTA's partial (O unnormalised w.r.t. M, M, Lambda).
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, dim = idx - (idx / D) * D;
    float a = 0.f;
#pragma unroll 4
    for (int q = 0; q < NGRP; ++q) a = fmaf(sm_acc[(q * G + g) * D + dim], sm_fac[q * G + g], a);
    const int64_t pidx = wk.pbase + (int64_t)(h0 + g) * wk.wtot + wk.slot;
    __stcg(p.part_o + pidx * D + dim, a);
  }
  if (tid < G) {
    const int64_t pidx = wk.pbase + (int64_t)(h0 + tid) * wk.wtot + wk.slot;
    __stcg(p.part_m + pidx, sm_ML[2 * tid]);
    __stcg(p.part_l + pidx, sm_ML[2 * tid + 1]);
  }
  if (MODE == 1) return;

  // Arrival: data first, then the counter (release); the last arriver acquires.
  __threadfence();
  __syncthreads();
  uint32_t* cnt = p.counters + (int64_t)wk.b * p.Hkv + wk.kvh;
  if (tid == 0) {
    const uint32_t old = atom_add_acq_rel_gpu(cnt, 1u);
    if (old >= (uint32_t)wk.wtot) atomicOr(p.status, kStatusCounter);
    sm_last = (old == (uint32_t)(wk.wtot - 1));
  }
  __syncthreads();
  if (!sm_last) return;
  __threadfence();
  combine_partials<T, D, G>(p, wk.b, wk.kvh, wk.wtot, wk.pbase, reinterpret_cast<float*>(smem));
  if (tid == 0) *cnt = 0u;
}

// Two-launch ablation, second kernel: one CTA per (sequence, KV head) combines
// the partials written by fd_split_kernel<..., 1>.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 2) fd_combine_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int b = blockIdx.x / p.Hkv, kvh = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
  const int wtot = (p.unit_base[b + 1] - p.unit_base[b]) / p.Hkv;
  const int64_t pbase = (int64_t)(p.unit_base[b] / p.Hkv) * p.Hq;
  combine_partials<T, D, G>(p, b, kvh, wtot, pbase, reinterpret_cast<float*>(smem));
}

}  // namespace dev

template <typename T, int D, int G>
cudaError_t launch_dg(const Params& p, int mode, int grid, cudaStream_t stream) {
  const size_t smem = smem_bytes_for(D);
  const void* fn;
  if (mode == 0) fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, 0>);
  else if (mode == 1) fn = reinterpret_cast<const void*>(&dev::fd_split_kernel<T, D, G, 1>);
  else fn = reinterpret_cast<const void*>(&dev::fd_combine_kernel<T, D, G>);
  int dev_id = 0;
  cudaError_t err = cudaGetDevice(&dev_id);
  if (err != cudaSuccess) return err;
  // The opt-in shared-memory size is a per-device function attribute.
  static uint64_t done_mask[3] = {0, 0, 0};
  const uint64_t bit = 1ull << (dev_id & 63);
  if (!(__atomic_load_n(&done_mask[mode], __ATOMIC_ACQUIRE) & bit)) {
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    __atomic_fetch_or(&done_mask[mode], bit, __ATOMIC_RELEASE);
  }
  void* args[] = {const_cast<Params*>(&p)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, smem, stream);
}

template <typename T>
cudaError_t launch_typed(const Params& p, int d, int G, int mode, int grid, cudaStream_t s) {
#define FD_CASE(DD, GG) \
  if (d == DD && G == GG) return launch_dg<T, DD, GG>(p, mode, grid, s);
  FD_CASE(64, 1) FD_CASE(64, 2) FD_CASE(64, 4) FD_CASE(64, 8)
  FD_CASE(128, 1) FD_CASE(128, 2) FD_CASE(128, 4) FD_CASE(128, 8)
#undef FD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fd
