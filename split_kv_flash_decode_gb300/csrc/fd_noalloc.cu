// fd_decode_noalloc: the fused decode with its scratch in a static device array.
//
// Some callers cannot allocate device memory at the moment they decode: code
// running inside an engine or framework that owns the device allocator and
// forbids raw cudaMalloc (a plugin's enqueue, a caching-allocator arena that
// must not fragment), or a call made where an allocation would synchronise
// the device.  This entry point needs no workspace from them: the arrival
// counters, status word and fp32 partials live in one file-scope __device__
// array of FD_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library
// holds until the process exits.  It calls no cudaMalloc, cudaFree or other
// allocating routine.
#include <mutex>

#include "fd_plan_internal.h"

namespace {

// The scratch array.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) on the first call made on it.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return FD_ERR_CUDA;
    }
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return FD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fd_decode_noalloc(fd_plan_t pl, const void* q, const void* k, const void* v,
                                 void* out, float* lse, cudaStream_t stream) {
  if (!pl || !q || !out) return FD_ERR_INVALID;
  if (pl->page_size != 0) return FD_ERR_INVALID;  // contiguous K/V only
  if (pl->n_tokens > 0 && (!k || !v)) return FD_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return FD_ERR_ALIGN;
  // The plan's scratch (counters, status, partials) must fit in the static array.
  if (pl->ws_bytes > (size_t)FD_NOALLOC_SCRATCH_BYTES) return FD_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != FD_OK) return rc;

  fd::Params p = pl->params;
  if (pl->n_tokens > 0) {
    rc = fd::encode_kv_map(&p.tm_k, k, pl->n_tokens, p.box_rows, pl);
    if (rc == FD_OK) rc = fd::encode_kv_map(&p.tm_v, v, pl->n_tokens, p.box_rows, pl);
    if (rc != FD_OK) return rc;
  }
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<uint32_t*>(ws + pl->off_counters);
  p.part = reinterpret_cast<float*>(ws + pl->off_part);
  p.flags = reinterpret_cast<uint32_t*>(ws + pl->off_flags);
  p.drop_flag = (pl->flags & FD_PLAN_TEST_DROP_FLAG) ? 1 : 0;

  // The array keeps whatever the previous call left: the status word and the
  // arrival counters must start at zero, so clear them on the stream first.
  cudaError_t err = cudaMemsetAsync(ws, 0, pl->off_part, stream);
  if (err == cudaSuccess) {
    auto launch = pl->dtype == FD_BF16 ? fd::launch_bf16 : fd::launch_f16;
    const bool pdl = !(pl->flags & FD_PLAN_NO_PDL);
    if (pl->flags & FD_PLAN_TWO_LAUNCH) {
      err = launch(p, pl->d, pl->G, pl->path, 1, pdl, pl->ctas, stream);
      if (err == cudaSuccess)
        err = launch(p, pl->d, pl->G, pl->path, 2, pdl, pl->B * pl->Hkv, stream);
    } else {
      err = launch(p, pl->d, pl->G, pl->path, (pl->flags & FD_PLAN_WAITS) ? 3 : 0, pdl, pl->ctas,
                   stream);
    }
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return err == cudaErrorCooperativeLaunchTooLarge ? FD_ERR_UNSUPPORTED : FD_ERR_CUDA;
  }
  return FD_OK;
}
