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
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>  // PFN_cuCtxGetCurrent, PFN_cuCtxGetId

#include "fd_plan_internal.h"

namespace {

// The scratch array.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchSlot {
  unsigned long long ctx_id;  // driver id of the context the address belongs to
  void* addr;
};
ScratchSlot g_scratch[kMaxDevices] = {};

// Driver calls that name the current context: its unique id changes when the
// context is destroyed and created again (cudaDeviceReset), even if the handle
// value is reused, and the module holding the array is then loaded again.
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
  });
  return fns;
}

// Id of the calling thread's current context; 0 if there is none yet.
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!f.get_current || !f.get_id || f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      f.get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array in the current device's context.  It is
// looked up (cudaGetSymbolAddress, with that device current) on the first call in
// each context, and kept for later calls in the same context.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long id = current_ctx_id();
  if (id == 0 || g_scratch[dev].addr == nullptr || g_scratch[dev].ctx_id != id) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return FD_ERR_CUDA;
    }
    g_scratch[dev].addr = addr;
    g_scratch[dev].ctx_id = current_ctx_id();  // the lookup made the context current
  }
  *out = g_scratch[dev].addr;
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

  // The array keeps whatever the previous call left: the status word and the
  // arrival counters must start at zero, so clear them on the stream first.
  cudaError_t err = cudaMemsetAsync(ws, 0, pl->off_part, stream);
  if (err == cudaSuccess) {
    if (pl->flags & FD_PLAN_TWO_LAUNCH) {
      err = fd::launch_plan(pl, p, 1, pl->ctas, stream);
      if (err == cudaSuccess) err = fd::launch_plan(pl, p, 2, pl->B * pl->Hkv, stream);
    } else {
      err = fd::launch_plan(pl, p, fd::fused_mode(pl), pl->ctas, stream);
    }
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fd::launch_status(err);
  }
  if (pl->flags & FD_PLAN_DEBUG) {
    int32_t st = FD_OK;
    rc = fd_noalloc_status(pl, stream, &st);
    if (rc != FD_OK) return rc;
    if (st != FD_OK) return st;
  }
  return FD_OK;
}

// Status of the last fd_decode_noalloc call of this plan's shape on the current
// device: the status word, then the counters and ready flags, which a completed
// decode leaves at zero.  Reads through the runtime (device-to-host copies into
// stack buffers); allocates nothing.
extern "C" int fd_noalloc_status(fd_plan_t pl, cudaStream_t stream, int32_t* status) {
  if (!pl || !status) return FD_ERR_INVALID;
  if (pl->ws_bytes > (size_t)FD_NOALLOC_SCRATCH_BYTES) return FD_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != FD_OK) return rc;
  const uint8_t* ws = static_cast<const uint8_t*>(scratch);
  uint32_t word = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return FD_ERR_CUDA;
  }
  // Counters and flags: [off_counters, off_part) holds both (flags follow the counters).
  bool at_rest = true;
  uint32_t buf[1024];
  for (size_t off = pl->off_counters; off < pl->off_part && at_rest; off += sizeof(buf)) {
    const size_t n = std::min(sizeof(buf), pl->off_part - off);
    if (cudaMemcpy(buf, ws + off, n, cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return FD_ERR_CUDA;
    }
    for (size_t i = 0; i < n / sizeof(uint32_t); ++i) at_rest = at_rest && buf[i] == 0u;
  }
  if (cudaMemset(const_cast<uint8_t*>(ws), 0, sizeof(word)) != cudaSuccess) {
    cudaGetLastError();
    return FD_ERR_CUDA;
  }
  *status = (word & fd::kStatusTimeout) ? FD_ERR_TIMEOUT
          : (word != 0 || !at_rest)     ? FD_ERR_STATE
                                        : FD_OK;
  return FD_OK;
}
