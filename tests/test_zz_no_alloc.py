"""fd_decode_noalloc: the entry point for callers that cannot allocate device memory.

Code that runs inside an engine owning the device allocator (a plugin enqueue
where cudaMalloc is not allowed, an arena that must not fragment) cannot hand
fd_decode a workspace.  fd_decode_noalloc keeps that scratch in the library's
static device array instead.  The GPU test calls it through the C ABI twice in
a row and compares each result with fd_decode's (the workspace entry point),
within the parity tolerances.  This file is collected last so that a run that
stops at the first failure has run every other test first.
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


def test_noalloc_rejects_plans_beyond_the_static_scratch():
    """No CUDA call is made: the size check comes first."""
    fd = _fd()
    plan = fd.fd_plan(256, 64, 8, 128, [4096] * 256, 16, "f16", num_sms=152)
    assert plan.workspace_bytes > fd.FD_NOALLOC_SCRATCH_BYTES
    rc = fd.lib().fd_decode_noalloc(plan.handle, 256, 256, 256, 256, 0, None)
    assert rc == fd.FD_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_matches_fd_decode_on_two_calls_in_a_row():
    import torch
    fd = _fd()
    p = workloads.gqa4_d128_L32k_W8()
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype)
    assert dec.plan.workspace_bytes <= fd.FD_NOALLOC_SCRATCH_BYTES
    q, k, v = (torch.from_numpy(x).cuda() for x in (p.q, p.k, p.v))
    ref_out, ref_lse = dec(q, k, v)                      # fd_decode with a caller workspace
    torch.cuda.synchronize()
    ref_out = ref_out.double().cpu().numpy()
    ref_lse = ref_lse.double().cpu().numpy()
    L = fd.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((p.B, p.Hq), float("nan"), dtype=torch.float32, device="cuda")
        rc = L.fd_decode_noalloc(dec.plan.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 out.data_ptr(), lse.data_ptr(), ctypes.c_void_p(stream))
        assert rc == fd.FD_OK, fd.fd_strerror(rc)
        torch.cuda.synchronize()
        o = out.double().cpu().numpy()
        l = lse.double().cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all(), f"call {call}: output not written"
        assert np.abs(o - ref_out).max() <= OUT_TOL, f"call {call}"
        assert np.abs(l - ref_lse).max() <= LSE_TOL, f"call {call}"
