"""fd_decode_noalloc: the entry point for callers that cannot allocate device memory.

Code that runs inside an engine owning the device allocator (a plugin enqueue
where cudaMalloc is not allowed, an arena that must not fragment) cannot hand
fd_decode a workspace.  fd_decode_noalloc keeps that scratch in the library's
static device array instead, and fd_noalloc_status reads that array's status.

The GPU tests call both through the C ABI.  Every variant of the kernel that
the entry point can launch (f16, bf16, two launches, the in-cluster segment
merge, an FP8 cache, fine-grained waits, the combine inside a cluster per
(sequence, KV head), tcgen05 consumers) is compared with fd_decode (the
workspace entry point) on the same plan and inputs, on two calls in a row that
follow a call with a different plan (the array keeps the previous call's
partials).  The deterministic variants must match bit for bit; the
fine-grained-waits variant combines in arrival order and is held to the parity
tolerances.  After every call the status reader must find the counters and
flags back at zero.  This file is collected last so that a run that stops at the
first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest

import workloads

OUT_TOL = 2e-3
LSE_TOL = 1e-4


def _fd():
    import split_kv_flash_decode_gb300 as fd
    from split_kv_flash_decode_gb300 import build
    build.build()
    return fd


def _to_torch(x, dtype):
    import torch
    if x.dtype == np.uint8 or dtype == "f16":          # uint8: FP8 E4M3 codes
        t = torch.from_numpy(np.ascontiguousarray(x))
    else:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def _plan_dtype(p):
    return "f16_e4m3kv" if p.kv_type == "e4m3" else p.dtype


def _noalloc(fd, plan, q, k, v, out, lse):
    """One fd_decode_noalloc call through the raw C ABI on torch's current stream."""
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    return fd.lib().fd_decode_noalloc(plan.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                      out.data_ptr(), 0 if lse is None else lse.data_ptr(),
                                      ctypes.c_void_p(stream))


def _status(fd, plan):
    import torch
    st = ctypes.c_int32(99)
    rc = fd.lib().fd_noalloc_status(plan.handle,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                    ctypes.byref(st))
    assert rc == fd.FD_OK, fd.fd_strerror(rc)
    return st.value


def test_noalloc_rejects_plans_beyond_the_static_scratch():
    """No CUDA call is made: the size check comes first."""
    fd = _fd()
    plan = fd.fd_plan(256, 64, 8, 128, [4096] * 256, 16, "f16", num_sms=152)
    assert plan.workspace_bytes > fd.FD_NOALLOC_SCRATCH_BYTES
    rc = fd.lib().fd_decode_noalloc(plan.handle, 256, 256, 256, 256, 0, None)
    assert rc == fd.FD_ERR_UNSUPPORTED
    st = ctypes.c_int32(0)
    assert fd.lib().fd_noalloc_status(plan.handle, None, ctypes.byref(st)) == fd.FD_ERR_UNSUPPORTED
    assert fd.lib().fd_noalloc_status(None, None, ctypes.byref(st)) == fd.FD_ERR_INVALID


def _small(dtype, seed, G=4):
    return workloads.make_problem("noalloc", 3, 8 * G, 8, 128, [9000, 17, 4096], [4, 2, 8], dtype,
                                  seed=seed)


def _variants(fd):
    return {
        "f16_32k": (workloads.gqa4_d128_L32k_W8, 0),
        "bf16": (lambda: _small("bf16", 91), 0),
        "two_launch": (lambda: _small("bf16", 92), fd.FD_PLAN_TWO_LAUNCH),
        "cluster": (lambda: _small("f16", 93, G=8), fd.FD_PLAN_CLUSTER),
        "e4m3_kv": (lambda: workloads.with_e4m3_kv(_small("f16", 94)), 0),
        "waits": (lambda: _small("f16", 95), fd.FD_PLAN_WAITS),
        "cluster_combine": (lambda: workloads.make_problem("noalloc_cc", 3, 32, 8, 128,
                                                           [9000, 17, 4096], 4, "bf16", seed=98),
                            fd.FD_PLAN_CLUSTER_COMBINE),
        "tcgen05": (lambda: _small("f16", 99, G=16), fd.FD_PLAN_TCGEN05),
    }


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["f16_32k", "bf16", "two_launch", "cluster", "e4m3_kv", "waits",
                                     "cluster_combine", "tcgen05"])
def test_noalloc_matches_fd_decode_on_two_calls_in_a_row(variant):
    import torch
    fd = _fd()
    make, flags = _variants(fd)[variant]
    p = make()
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, _plan_dtype(p), flags=flags)
    assert dec.plan.workspace_bytes <= fd.FD_NOALLOC_SCRATCH_BYTES
    q = _to_torch(p.q, p.dtype)
    k, v = _to_torch(p.k, p.dtype), _to_torch(p.v, p.dtype)
    ref_out, ref_lse = dec(q, k, v)                      # fd_decode with a caller workspace
    assert dec.status() == fd.FD_OK
    ref_out = ref_out.double().cpu().numpy()
    ref_lse = ref_lse.double().cpu().numpy()

    # A call with a different plan first: it leaves its own partials in the array.
    o = workloads.make_problem("noalloc_other", 2, 64, 8, 128, [20000, 5000], [8, 3], "f16",
                               seed=96)
    other = fd.fd_plan(o.B, o.Hq, o.Hkv, o.d, o.seqlens, o.W, "f16")
    oq, ok_, ov = _to_torch(o.q, "f16"), _to_torch(o.k, "f16"), _to_torch(o.v, "f16")
    oo = torch.empty_like(oq)
    ol = torch.empty((o.B, o.Hq), dtype=torch.float32, device="cuda")
    assert _noalloc(fd, other, oq, ok_, ov, oo, ol) == fd.FD_OK
    assert _status(fd, other) == fd.FD_OK

    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((p.B, p.Hq), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(fd, dec.plan, q, k, v, out, lse)
        assert rc == fd.FD_OK, fd.fd_strerror(rc)
        assert _status(fd, dec.plan) == fd.FD_OK, f"call {call}: counters or status not at rest"
        got_o = out.double().cpu().numpy()
        got_l = lse.double().cpu().numpy()
        assert not np.isnan(got_o).any() and not np.isnan(got_l).any(), f"call {call}: not written"
        if flags & fd.FD_PLAN_WAITS:
            full = ~np.isneginf(ref_lse)
            assert np.array_equal(np.isneginf(got_l), ~full)
            assert np.abs(got_o - ref_out).max() <= OUT_TOL, f"call {call}"
            assert np.abs(got_l[full] - ref_lse[full]).max() <= LSE_TOL, f"call {call}"
        else:
            assert np.array_equal(got_o, ref_out), f"call {call}: out differs from fd_decode"
            assert np.array_equal(got_l, ref_lse), f"call {call}: lse differs from fd_decode"


@pytest.mark.gpu
def test_noalloc_reports_a_bounded_wait_that_ran_out():
    """A ready flag that nothing sets: the status reader reports FD_ERR_TIMEOUT, and the
    next call, with a clean plan of the same shape, reports FD_OK and is correct."""
    import torch
    fd = _fd()
    p = _small("f16", 97)
    q, k, v = (_to_torch(x, "f16") for x in (p.q, p.k, p.v))
    hooked = fd.fd_plan(p.B, p.Hq, p.Hkv, p.d, p.seqlens, p.W, "f16",
                        flags=fd.FD_PLAN_WAITS | fd.FD_PLAN_TEST_DROP_FLAG)
    out = torch.empty_like(q)
    lse = torch.empty((p.B, p.Hq), dtype=torch.float32, device="cuda")
    assert _noalloc(fd, hooked, q, k, v, out, lse) == fd.FD_OK
    assert _status(fd, hooked) == fd.FD_ERR_TIMEOUT
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, "f16", flags=fd.FD_PLAN_WAITS)
    ref_out, ref_lse = dec(q, k, v)
    assert _noalloc(fd, dec.plan, q, k, v, out, lse) == fd.FD_OK
    assert _status(fd, dec.plan) == fd.FD_OK
    assert (out.double() - ref_out.double()).abs().max().item() <= OUT_TOL
    assert (lse.double() - ref_lse.double()).abs().max().item() <= LSE_TOL
