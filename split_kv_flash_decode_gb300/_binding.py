"""ctypes binding of libfd_gb300.so: argument marshalling only.

Every function here forwards to the C entry point of the same name in
``include/fd.h``; all compute runs in the library's CUDA kernels.  PyTorch
supplies device memory and streams.  If the library is missing the calls raise
-- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libfd_gb300.so")

FD_OK = 0
FD_ERR_INVALID = -1
FD_ERR_UNSUPPORTED = -2
FD_ERR_ALIGN = -3
FD_ERR_CUDA = -4
FD_ERR_NOMEM = -5
FD_ERR_STATE = -6
FD_ERR_TIMEOUT = -7

FD_F16 = 0
FD_BF16 = 1
FD_F16_E4M3KV = 2
FD_PLAN_LITERAL_W = 0x1
FD_PLAN_DEBUG = 0x2
FD_PLAN_TWO_LAUNCH = 0x4
FD_PLAN_FFMA = 0x8
FD_PLAN_NO_PDL = 0x10
FD_PLAN_WAITS = 0x20
FD_PLAN_TEST_DROP_FLAG = 0x40
FD_PLAN_NO_CLUSTER = 0x80
FD_PLAN_CLUSTER = 0x100
FD_PLAN_TEST_SKIP_TILE = 0x200
FD_PLAN_TCGEN05 = 0x400
FD_PLAN_CLUSTER_COMBINE = 0x800
FD_PLAN_MMA_SYNC = 0x1000
FD_PLAN_TEST_DROP_ARRIVAL = 0x2000
FD_PLAN_DEEP_RING = 0x4000
FD_PLAN_COMBINERS_SHIFT = 16
FD_PLAN_COMBINERS_MASK = 7 << FD_PLAN_COMBINERS_SHIFT
# FD_PLAN_COMBINERS[n]: at most n CTAs share the combine of one (sequence, KV head) pair.
FD_PLAN_COMBINERS = {n: (k + 1) << FD_PLAN_COMBINERS_SHIFT for k, n in enumerate((1, 2, 4, 8, 16))}
FD_PLAN_SINGLE_COMBINER = FD_PLAN_COMBINERS[1]
FD_MAX_BATCH = 256
FD_MAX_PARTIALS = 1024

DTYPES = {"f16": FD_F16, "bf16": FD_BF16, "f16_e4m3kv": FD_F16_E4M3KV}

# Every symbol include/fd.h declares.
EXPORTED = (
    "fd_plan", "fd_plan_destroy", "fd_workspace_bytes", "fd_workspace_init", "fd_decode",
    "fd_workspace_status", "fd_strerror", "fd_plan_get_info", "fd_plan_get_range", "fd_version",
    "fd_decode_noalloc", "fd_noalloc_status", "fd_plan_paged", "fd_decode_paged",
)
FD_NOALLOC_SCRATCH_BYTES = 32 << 20


class FdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})")


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32), ("G", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32), ("chunks", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("ctas", ctypes.c_int32), ("max_partials", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64), ("total_partials", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_uint64), ("kv_bytes", ctypes.c_uint64),
        ("path", ctypes.c_int32), ("records_per_segment", ctypes.c_int32),
        ("combine_cluster", ctypes.c_int32), ("combiners", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with split_kv_flash_decode_gb300.build.build()"
                    " (nvcc, sm_103a); there is no fallback implementation")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
            L.fd_plan.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.c_int, u32,
                                  ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)]
            L.fd_plan.restype = ctypes.c_int
            L.fd_plan_destroy.argtypes = [vp]
            L.fd_plan_destroy.restype = ctypes.c_int
            L.fd_workspace_bytes.argtypes = [vp]
            L.fd_workspace_bytes.restype = sz
            L.fd_workspace_init.argtypes = [vp, vp, vp]
            L.fd_workspace_init.restype = ctypes.c_int
            L.fd_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
            L.fd_decode.restype = ctypes.c_int
            L.fd_workspace_status.argtypes = [vp, vp, vp, ctypes.POINTER(i32)]
            L.fd_workspace_status.restype = ctypes.c_int
            L.fd_strerror.argtypes = [ctypes.c_int]
            L.fd_strerror.restype = ctypes.c_char_p
            L.fd_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
            L.fd_plan_get_info.restype = ctypes.c_int
            L.fd_plan_get_range.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(i32),
                                            ctypes.POINTER(i32)]
            L.fd_plan_get_range.restype = ctypes.c_int
            L.fd_plan_paged.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.c_int,
                                        ctypes.c_int, u32, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(vp)]
            L.fd_plan_paged.restype = ctypes.c_int
            L.fd_decode_paged.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp,
                                          vp, vp]
            L.fd_decode_paged.restype = ctypes.c_int
            L.fd_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            L.fd_decode_noalloc.restype = ctypes.c_int
            L.fd_noalloc_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
            L.fd_noalloc_status.restype = ctypes.c_int
            L.fd_version.argtypes = []
            L.fd_version.restype = ctypes.c_int
            _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().fd_strerror(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != FD_OK:
        raise FdError(rc, where)


def _i32_array(values, n: int):
    arr = (ctypes.c_int32 * n)()
    vals = list(values)
    for i in range(n):
        arr[i] = int(vals[i])
    return arr


def _ptr(t) -> int:
    """Device address of a tensor (or an int address, or None -> 0)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class Plan:
    """Owns one fd_plan_t handle (fd_plan_destroy on close / garbage collection)."""

    def __init__(self, handle: int):
        self.handle = handle
        info = PlanInfo()
        _check(lib().fd_plan_get_info(handle, ctypes.byref(info)), "fd_plan_get_info")
        self.info = {name: getattr(info, name) for name, _ in PlanInfo._fields_}

    @property
    def workspace_bytes(self) -> int:
        return fd_workspace_bytes(self)

    def range(self, b: int, slot: int):
        return fd_plan_get_range(self, b, slot)

    def close(self) -> None:
        if self.handle:
            lib().fd_plan_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fd_plan(B, Hq, Hkv, d, seqlens, W, dtype="f16", flags=0, chunks=0, num_sms=0) -> Plan:
    """fd_plan: validate a decode shape and build its work decomposition (host only)."""
    seqlens = list(seqlens)
    W = [W] * B if isinstance(W, int) else list(W)
    if len(seqlens) != B or len(W) != B:
        raise FdError(FD_ERR_INVALID, "fd_plan: seqlens and W need B entries")
    handle = ctypes.c_void_p()
    rc = lib().fd_plan(int(B), int(Hq), int(Hkv), int(d), _i32_array(seqlens, B),
                       _i32_array(W, B), DTYPES[dtype] if isinstance(dtype, str) else int(dtype),
                       int(flags), int(chunks), int(num_sms), ctypes.byref(handle))
    _check(rc, "fd_plan")
    return Plan(handle.value)


def fd_plan_paged(B, Hq, Hkv, d, seqlens, W, page_size, dtype="f16", flags=0, chunks=0,
                  num_sms=0) -> Plan:
    """fd_plan_paged: plan a decode over a paged KV cache (host only)."""
    seqlens = list(seqlens)
    W = [W] * B if isinstance(W, int) else list(W)
    if len(seqlens) != B or len(W) != B:
        raise FdError(FD_ERR_INVALID, "fd_plan_paged: seqlens and W need B entries")
    handle = ctypes.c_void_p()
    rc = lib().fd_plan_paged(int(B), int(Hq), int(Hkv), int(d), _i32_array(seqlens, B),
                             _i32_array(W, B), int(page_size),
                             DTYPES[dtype] if isinstance(dtype, str) else int(dtype), int(flags),
                             int(chunks), int(num_sms), ctypes.byref(handle))
    _check(rc, "fd_plan_paged")
    return Plan(handle.value)


def fd_decode_paged(plan: Plan, q, k_pages, v_pages, num_pages, block_table, bt_stride, out, lse,
                    workspace, stream=None) -> None:
    """fd_decode_paged: the fused decode over a paged cache (block tables)."""
    _check(lib().fd_decode_paged(plan.handle, _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                 int(num_pages), _ptr(block_table), int(bt_stride), _ptr(out),
                                 _ptr(lse), _ptr(workspace), _stream(stream)), "fd_decode_paged")


def fd_plan_destroy(plan: Plan) -> None:
    plan.close()


def fd_workspace_bytes(plan: Plan) -> int:
    return int(lib().fd_workspace_bytes(plan.handle))


def fd_workspace_init(plan: Plan, workspace, stream=None) -> None:
    _check(lib().fd_workspace_init(plan.handle, _ptr(workspace), _stream(stream)),
           "fd_workspace_init")


def fd_decode(plan: Plan, q, k, v, out, lse, workspace, stream=None) -> None:
    """fd_decode: one fused launch on `stream` (default: torch's current stream)."""
    _check(lib().fd_decode(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                           _ptr(workspace), _stream(stream)), "fd_decode")


def fd_decode_noalloc(plan: Plan, q, k, v, out, lse, stream=None) -> None:
    """fd_decode_noalloc: the fused decode with the library's static device scratch
    (for callers that cannot allocate device memory; see include/fd.h)."""
    _check(lib().fd_decode_noalloc(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                   _stream(stream)), "fd_decode_noalloc")


def fd_noalloc_status(plan: Plan, stream=None) -> int:
    """fd_noalloc_status: status of the last fd_decode_noalloc call (synchronises)."""
    st = ctypes.c_int32(0)
    _check(lib().fd_noalloc_status(plan.handle, _stream(stream), ctypes.byref(st)),
           "fd_noalloc_status")
    return st.value


def fd_workspace_status(plan: Plan, workspace, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(lib().fd_workspace_status(plan.handle, _ptr(workspace), _stream(stream),
                                     ctypes.byref(st)), "fd_workspace_status")
    return st.value


def fd_plan_get_range(plan: Plan, b: int, slot: int):
    lo, hi = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().fd_plan_get_range(plan.handle, int(b), int(slot), ctypes.byref(lo),
                                   ctypes.byref(hi)), "fd_plan_get_range")
    return lo.value, hi.value


def fd_version() -> int:
    return int(lib().fd_version())
