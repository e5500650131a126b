"""Host-side tests of the C ABI (no GPU needed: no compute call is made).

They check that the library loads and exports every entry point include/fd.h
declares, that fd_plan validates its arguments with the documented status
codes, and that the work decomposition tiles every sequence exactly: each
chunk lies inside the segment of the oracle's segment rule, chunks are disjoint
and cover [0, L_b).
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import split_kv_flash_decode_gb300 as fd
from split_kv_flash_decode_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd.h")


@pytest.fixture(scope="module", autouse=True)
def built_lib():
    build.build()
    return fd.lib()


def declared_entry_points():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z_]+)\s*\(", text)))


def test_header_declares_what_binding_exports():
    decl = declared_entry_points()
    assert decl == sorted(_binding.EXPORTED)


def test_library_exports_every_declared_symbol():
    so = ctypes.CDLL(_binding.LIB_PATH)
    for name in declared_entry_points():
        assert hasattr(so, name), name


def test_version_and_strerror():
    assert fd.fd_version() == 0x000100
    for code in (fd.FD_OK, fd.FD_ERR_INVALID, fd.FD_ERR_UNSUPPORTED, fd.FD_ERR_ALIGN,
                 fd.FD_ERR_CUDA, fd.FD_ERR_NOMEM, fd.FD_ERR_STATE, fd.FD_ERR_TIMEOUT):
        s = fd.fd_strerror(code)
        assert s.startswith("FD_")
    assert "unknown" in fd.fd_strerror(12345)


def _raw_plan(B, Hq, Hkv, d, seqlens, W, dtype=0, flags=0, chunks=0, num_sms=152):
    L = fd.lib()
    arr = (ctypes.c_int32 * max(1, len(seqlens)))(*seqlens)
    warr = (ctypes.c_int32 * max(1, len(W)))(*W)
    h = ctypes.c_void_p()
    rc = L.fd_plan(B, Hq, Hkv, d, arr, warr, dtype, flags, chunks, num_sms, ctypes.byref(h))
    if rc == 0:
        L.fd_plan_destroy(h)
    return rc


@pytest.mark.parametrize("args,code", [
    ((0, 8, 8, 128, [], []), fd.FD_ERR_INVALID),                      # B < 1
    ((1, 8, 3, 128, [10], [1]), fd.FD_ERR_INVALID),                   # Hq % Hkv
    ((1, 8, 8, 128, [-1], [1]), fd.FD_ERR_INVALID),                   # negative length
    ((1, 8, 8, 128, [10], [0]), fd.FD_ERR_INVALID),                   # W < 1
    ((1, 8, 8, 96, [10], [1]), fd.FD_ERR_UNSUPPORTED),                # d
    ((1, 24, 8, 128, [10], [1]), fd.FD_ERR_UNSUPPORTED),              # G = 3
    ((1, 256, 8, 128, [10], [1]), fd.FD_ERR_UNSUPPORTED),             # G = 32
    ((1, 128, 8, 128, [10], [1]), fd.FD_OK),                          # G = 16 (tensor cores)
    ((257, 8, 8, 128, [1] * 257, [1] * 257), fd.FD_ERR_UNSUPPORTED),  # batch limit
    ((1, 8, 8, 128, [10], [1025]), fd.FD_ERR_UNSUPPORTED),            # partial limit
    ((1, 8, 8, 128, [10], [1]), fd.FD_OK),
])
def test_plan_validation(args, code):
    assert _raw_plan(*args) == code


def test_plan_bad_dtype_flags_chunks():
    assert _raw_plan(1, 8, 8, 128, [10], [1], dtype=3) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [1], dtype=2) == fd.FD_ERR_UNSUPPORTED  # FP8 K/V: G >= 4
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=0x80000) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=6 << 16) == fd.FD_ERR_INVALID  # cap code 6
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_CLUSTER | fd.FD_PLAN_NO_CLUSTER) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_CLUSTER | fd.FD_PLAN_WAITS) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [1], chunks=-1) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [600], chunks=2) == fd.FD_ERR_UNSUPPORTED
    # flag combinations
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_WAITS | fd.FD_PLAN_TWO_LAUNCH) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_TEST_DROP_FLAG) == fd.FD_ERR_INVALID
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_WAITS | fd.FD_PLAN_TEST_DROP_FLAG) == fd.FD_OK
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_TEST_SKIP_TILE) == fd.FD_OK
    assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_WAITS | fd.FD_PLAN_TEST_DROP_FLAG
                     | fd.FD_PLAN_TEST_SKIP_TILE) == fd.FD_ERR_INVALID
    L = fd.lib()
    assert L.fd_plan(1, 8, 8, 128, None, None, 0, 0, 0, 152, None) == fd.FD_ERR_INVALID
    assert L.fd_plan_destroy(None) == fd.FD_OK
    assert L.fd_workspace_bytes(None) == 0


def test_null_pointer_rejections():
    p = fd.fd_plan(1, 8, 8, 64, [100], 4, "f16", num_sms=152)
    L = fd.lib()
    assert L.fd_decode(p.handle, None, None, None, None, None, None, None) == fd.FD_ERR_INVALID
    # misaligned device pointers are rejected before any CUDA call
    assert L.fd_decode(p.handle, 16, 16, 16, 16, 0, 8, None) == fd.FD_ERR_ALIGN
    assert L.fd_decode(p.handle, 24, 16, 16, 16, 0, 16, None) == fd.FD_ERR_ALIGN
    assert L.fd_workspace_init(p.handle, None, None) == fd.FD_ERR_INVALID
    assert L.fd_plan_get_info(None, None) == fd.FD_ERR_INVALID
    lo, hi = ctypes.c_int32(), ctypes.c_int32()
    assert L.fd_plan_get_range(p.handle, 1, 0, ctypes.byref(lo), ctypes.byref(hi)) == fd.FD_ERR_INVALID
    assert L.fd_plan_get_range(p.handle, 0, 4, ctypes.byref(lo), ctypes.byref(hi)) == fd.FD_ERR_INVALID


def _check_tiling(plan, seqlens, W):
    C = plan.info["chunks"]
    for b, L in enumerate(seqlens):
        segs = oracle.segment_bounds(int(L), int(W[b]))
        pos = 0
        for slot in range(int(W[b]) * C):
            lo, hi = plan.range(b, slot)
            s0, s1 = segs[slot // C]
            assert s0 <= lo <= hi <= s1, (b, slot, lo, hi, s0, s1)
            assert lo == pos, (b, slot)
            pos = hi
        assert pos == L


@pytest.mark.parametrize("seed", range(6))
def test_work_decomposition_tiles_sequences(seed):
    rs = np.random.default_rng(seed)
    B = int(rs.integers(1, 20))
    seqlens = rs.integers(0, 5000, size=B)
    seqlens[rs.integers(0, B)] = 0
    W = rs.integers(1, 40, size=B)
    for chunks in (0, 1, 3, 7):
        p = fd.fd_plan(B, 16, 4, 128, seqlens, W, "f16", chunks=chunks, num_sms=152)
        if chunks:
            assert p.info["chunks"] == chunks
        _check_tiling(p, seqlens, W)
        info = p.info
        assert info["ctas"] == 4 * int(W.sum()) * info["chunks"]
        assert info["total_partials"] == 16 * int(W.sum()) * info["chunks"]
        assert info["total_tokens"] == int(seqlens.sum())
        assert info["kv_bytes"] == int(seqlens.sum()) * 4 * 128 * 4


def test_literal_w_and_auto_chunks():
    # literal W: exactly W partials per sequence
    p = fd.fd_plan(64, 32, 8, 128, [8192] * 64, 16, "bf16", flags=fd.FD_PLAN_LITERAL_W,
                   chunks=5, num_sms=152)
    assert p.info["chunks"] == 1 and p.info["ctas"] == 64 * 8 * 16
    # auto: one wave of two CTAs per SM, segments not cut below 128 tokens
    p = fd.fd_plan(1, 32, 8, 128, [32768], 8, "f16", num_sms=152)
    assert p.info["chunks"] == 4 and p.info["ctas"] == 256
    p = fd.fd_plan(1, 8, 8, 64, [4096], 4, "f16", num_sms=152)
    assert p.info["chunks"] == 8  # 1024-token segments -> 128-token chunks, 256 CTAs
    p = fd.fd_plan(1, 8, 8, 64, [100], 4, "f16", num_sms=152)
    assert p.info["chunks"] == 1
    p = fd.fd_plan(1, 8, 8, 64, [2048], 4, "f16", num_sms=152)
    assert p.info["chunks"] == 4  # 512-token segments -> 128-token chunks, not 9 slots' worth


def test_records_per_segment():
    ring = {128: 96 * 1024, 64: 96 * 1024}   # K/V rings (bytes)

    def combiners(G, ctas, slots, partials):
        nc = min(G, 8) if ctas <= slots and G >= 8 else 1
        while nc > 1 and nc > partials:
            nc //= 2
        return nc
    # Auto: chunk records merge per segment (in a cluster of 2..8 CTAs) exactly when the
    # records one combiner reads, G / combiners * W * C * (d + 4) * 4 bytes, exceed the
    # ring (twice the ring over an FP8 cache).
    for Hq, W, chunks in ((32, 8, 2), (32, 8, 5), (32, 8, 8), (64, 8, 4), (128, 8, 4),
                          (128, 8, 9), (32, 8, 1), (64, 8, 16)):
        p = fd.fd_plan(1, Hq, 8, 128, [32768], W, "f16", chunks=chunks, num_sms=152)
        G = Hq // 8
        slots = 304                                         # mma.sync: two CTAs per SM
        nc = combiners(G, 8 * W * chunks, slots, W * chunks)
        multi = G // nc * W * chunks * 132 * 4 > ring[128]
        want = 1 if (multi and 2 <= chunks <= 8) else chunks
        assert p.info["chunks"] == chunks and p.info["records_per_segment"] == want, (Hq, chunks)
        assert p.info["combiners"] == (1 if want != chunks else nc), (Hq, chunks)
    # The default 32K GQA-4 and 128K GQA-8 plans fit one pass per combiner.
    assert fd.fd_plan(1, 32, 8, 128, [32768], 8, "f16", num_sms=152).info["records_per_segment"] == 4
    assert fd.fd_plan(1, 64, 8, 128, [131072], 8, "f16", num_sms=152).info["records_per_segment"] == 4
    fp8 = lambda Hq, f=0: fd.fd_plan(1, Hq, 8, 128, [131072], 8, "f16_e4m3kv", flags=f,  # noqa: E731
                                     num_sms=152)
    assert fp8(64).info["records_per_segment"] == 4 and fp8(128).info["records_per_segment"] == 4
    # One combiner: G * W * C * 528 bytes = 270 KB for G = 16 (> 2 rings), 135 KB for G = 8.
    assert fp8(64, fd.FD_PLAN_SINGLE_COMBINER).info["records_per_segment"] == 4
    assert fp8(128, fd.FD_PLAN_SINGLE_COMBINER).info["records_per_segment"] == 1
    p = fd.fd_plan(1, 32, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_CLUSTER, num_sms=152)
    assert p.info["chunks"] == 4 and p.info["records_per_segment"] == 1
    for flags in (fd.FD_PLAN_NO_CLUSTER, fd.FD_PLAN_WAITS):
        p = fd.fd_plan(1, 64, 8, 128, [131072], 8, "f16", flags=flags | fd.FD_PLAN_SINGLE_COMBINER,
                       num_sms=152)
        assert p.info["chunks"] == 4 and p.info["records_per_segment"] == 4
    # paged plans follow the same rule; one chunk per segment never forms a cluster
    p = fd.fd_plan_paged(1, 64, 8, 128, [131072], 8, 64, "f16", num_sms=152,
                         flags=fd.FD_PLAN_SINGLE_COMBINER)
    assert p.info["chunks"] == 4 and p.info["records_per_segment"] == 1
    p = fd.fd_plan_paged(1, 64, 8, 128, [131072], 8, 64, "f16", num_sms=152)
    assert p.info["records_per_segment"] == 4 and p.info["combiners"] == 8
    p = fd.fd_plan(1, 32, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_CLUSTER | fd.FD_PLAN_LITERAL_W,
                   num_sms=152)
    assert p.info["chunks"] == 1 and p.info["records_per_segment"] == 1
    # more than 8 chunks per segment cannot form a (portable) cluster
    p = fd.fd_plan(1, 32, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_CLUSTER, chunks=12,
                   num_sms=152)
    assert p.info["records_per_segment"] == 12


def test_consumer_path_choice():
    # tensor cores once the GQA group fills at least half of the mma N = 8 tile
    for G, path in ((1, 0), (2, 0), (4, 1), (8, 1)):
        p = fd.fd_plan(1, 8 * G, 8, 128, [1000], 2, "f16", num_sms=152)
        assert p.info["path"] == path, G
    p = fd.fd_plan(1, 64, 8, 128, [1000], 2, "bf16", flags=fd.FD_PLAN_FFMA, num_sms=152)
    assert p.info["path"] == 0
    # G = 16: mma.sync (two N tiles) unless tcgen05 is asked for
    assert fd.fd_plan(1, 128, 8, 128, [1000], 2, "f16", num_sms=152).info["path"] == 1
    assert fd.fd_plan(1, 128, 8, 128, [1000], 2, "f16", flags=fd.FD_PLAN_TCGEN05,
                      num_sms=152).info["path"] == 3
    assert fd.fd_plan(1, 128, 8, 128, [1000], 2, "bf16", flags=fd.FD_PLAN_MMA_SYNC,
                      num_sms=152).info["path"] == 1
    assert fd.fd_plan(1, 128, 8, 64, [1000], 2, "f16", num_sms=152).info["path"] == 1
    assert fd.fd_plan(1, 128, 8, 128, [1000], 2, "f16_e4m3kv", num_sms=152).info["path"] == 2
    with pytest.raises(fd.FdError) as ei:
        fd.fd_plan(1, 128, 8, 128, [1000], 2, "f16", flags=fd.FD_PLAN_FFMA, num_sms=152)
    assert ei.value.status == fd.FD_ERR_UNSUPPORTED
    assert _raw_plan(1, 32, 8, 128, [10], [1], flags=fd.FD_PLAN_MMA_SYNC | fd.FD_PLAN_FFMA) \
        == fd.FD_ERR_INVALID
    assert _raw_plan(1, 32, 8, 128, [10], [1], flags=fd.FD_PLAN_MMA_SYNC | fd.FD_PLAN_TCGEN05) \
        == fd.FD_ERR_UNSUPPORTED


def test_tcgen05_plan_rules():
    """tcgen05 consumers: d = 128, G in {4, 8, 16}, 16-bit K/V; paged caches align
    segments and chunks to its 128-token tiles."""
    for G in (4, 8, 16):
        for dtype in ("f16", "bf16"):
            p = fd.fd_plan(1, 8 * G, 8, 128, [1000], 2, dtype, flags=fd.FD_PLAN_TCGEN05,
                           num_sms=152)
            assert p.info["path"] == 3
    for Hq, d, dtype, flags in ((16, 128, "f16", 0), (8, 128, "bf16", 0), (32, 64, "f16", 0),
                                (32, 128, "f16_e4m3kv", 0), (32, 128, "f16", fd.FD_PLAN_FFMA)):
        with pytest.raises(fd.FdError) as ei:
            fd.fd_plan(1, Hq, 8, d, [4096], 4, dtype, flags=flags | fd.FD_PLAN_TCGEN05, num_sms=152)
        assert ei.value.status == fd.FD_ERR_UNSUPPORTED
    p = fd.fd_plan_paged(2, 32, 8, 128, [5000, 777], [3, 2], 16, "f16",
                         flags=fd.FD_PLAN_TCGEN05, num_sms=152)
    for b, L in ((0, 5000), (1, 777)):
        for slot in range(p.info["max_partials"] if b == 0 else 2 * p.info["chunks"]):
            lo, hi = p.range(b, slot)
            assert (lo % 128 == 0 or lo == L) and (hi % 128 == 0 or hi == L)


def test_cluster_combine_plan_rules():
    """FD_PLAN_CLUSTER_COMBINE: one cluster of W * C <= 16 CTAs per (sequence, KV head)."""
    p = fd.fd_plan(1, 32, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_CLUSTER_COMBINE, num_sms=152)
    assert p.info["chunks"] == 2 and p.info["combine_cluster"] == 16 and p.info["ctas"] == 128
    p = fd.fd_plan(64, 32, 8, 128, [8192] * 64, 16, "bf16",
                   flags=fd.FD_PLAN_CLUSTER_COMBINE | fd.FD_PLAN_LITERAL_W, num_sms=152)
    assert p.info["combine_cluster"] == 16 and p.info["ctas"] == 8192
    p = fd.fd_plan(2, 16, 4, 64, [300, 0], 3, "f16", flags=fd.FD_PLAN_CLUSTER_COMBINE, num_sms=152)
    assert p.info["combine_cluster"] == 3 * p.info["chunks"] <= 16
    assert fd.fd_plan(1, 32, 8, 128, [1000], 2, "f16", num_sms=152).info["combine_cluster"] == 0
    for W, chunks in (([4, 5], 0), ([17, 17], 0), ([8, 8], 3)):
        with pytest.raises(fd.FdError) as ei:      # ragged W, W > 16, W * C > 16
            fd.fd_plan(2, 32, 8, 128, [4096, 4096], W, "f16", flags=fd.FD_PLAN_CLUSTER_COMBINE,
                       chunks=chunks, num_sms=152)
        assert ei.value.status == fd.FD_ERR_UNSUPPORTED
    for other in (fd.FD_PLAN_WAITS, fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_CLUSTER, fd.FD_PLAN_NO_CLUSTER):
        assert _raw_plan(1, 8, 8, 128, [10], [1], flags=fd.FD_PLAN_CLUSTER_COMBINE | other) \
            == fd.FD_ERR_INVALID


def test_fp8_kv_plan_rules():
    p = fd.fd_plan(1, 32, 8, 128, [4096], 4, "f16_e4m3kv", num_sms=152)
    assert p.info["path"] == 2 and p.info["kv_bytes"] == 4096 * 8 * 128 * 2
    for Hq, d, flags in ((16, 128, 0), (32, 128, fd.FD_PLAN_FFMA), (32, 64, 0)):
        with pytest.raises(fd.FdError) as ei:
            fd.fd_plan(1, Hq, 8, d, [4096], 4, "f16_e4m3kv", flags=flags, num_sms=152)
        assert ei.value.status == fd.FD_ERR_UNSUPPORTED


def test_combine_scratch_limit():
    # The combine's coefficient scratch, (G * partials + 3 G) * 4 bytes, must fit the ring
    # it reuses; with a 96 KB ring even G = 16 with 1024 partials fits (66 KB), for the
    # fine-grained-waits variant too.
    fd.fd_plan(1, 128, 8, 64, [100000], 1024, "f16", flags=fd.FD_PLAN_LITERAL_W, num_sms=152)
    fd.fd_plan(1, 128, 8, 128, [100000], 1024, "f16", flags=fd.FD_PLAN_LITERAL_W | fd.FD_PLAN_WAITS,
               num_sms=152)
    with pytest.raises(fd.FdError) as ei:          # beyond the partial-record limit
        fd.fd_plan(1, 128, 8, 64, [100000], 1025, "f16", flags=fd.FD_PLAN_LITERAL_W, num_sms=152)
    assert ei.value.status == fd.FD_ERR_UNSUPPORTED


def test_workspace_layout():
    p = fd.fd_plan(3, 8, 2, 64, [10, 0, 700], [1, 2, 5], "f16", chunks=2, num_sms=152)
    P = 8 * (1 + 2 + 5) * 2
    assert p.info["total_partials"] == P
    need = 4 * 3 * 2 + 4 * p.info["ctas"] + 4 * P * (64 + 4)
    assert p.workspace_bytes >= need
    assert p.workspace_bytes % 256 == 0


def test_paged_plan_validation_and_alignment():
    L = fd.lib()
    arr = (ctypes.c_int32 * 2)(1000, 77)
    warr = (ctypes.c_int32 * 2)(3, 2)
    h = ctypes.c_void_p()
    for ps, code in ((0, fd.FD_ERR_INVALID), (8, fd.FD_ERR_UNSUPPORTED), (48, fd.FD_ERR_UNSUPPORTED),
                     (512, fd.FD_ERR_UNSUPPORTED), (16, fd.FD_OK), (256, fd.FD_OK)):
        rc = L.fd_plan_paged(2, 32, 8, 128, arr, warr, ps, 0, 0, 0, 152, ctypes.byref(h))
        assert rc == code, ps
        if rc == fd.FD_OK:
            L.fd_plan_destroy(h)
    for G, tile in ((4, 64), (1, 32)):
        p = fd.fd_plan_paged(2, 8 * G, 8, 128, [1000, 77], [3, 2], 16, "f16", chunks=3, num_sms=152)
        for b, Lb in enumerate((1000, 77)):
            pos = 0
            for slot in range((3, 2)[b] * 3):
                lo, hi = p.range(b, slot)
                assert lo == pos and hi >= lo and (lo % tile == 0 or lo == hi)
                pos = hi
            assert pos == Lb
        # contiguous decode entry point refuses paged plans (before any CUDA call)
        assert L.fd_decode(p.handle, 16, 16, 16, 16, 0, 16, None) == fd.FD_ERR_INVALID
        # short block-table stride
        need = -(-1000 // 16)
        assert L.fd_decode_paged(p.handle, 16, 16, 16, 100, 16, need - 1, 16, 0, 16, None) == fd.FD_ERR_INVALID
    c = fd.fd_plan(1, 8, 8, 64, [100], 1, "f16", num_sms=152)
    assert L.fd_decode_paged(c.handle, 16, 16, 16, 10, 16, 10, 16, 0, 16, None) == fd.FD_ERR_INVALID


def test_shared_combine_plan_rules():
    """The last arrivals of a pair share its combine by query heads only when the
    whole grid is resident at once, in the fused launch without clusters; the count
    is a power of two that divides G, at most the partials of the longest sequence."""
    def info(*a, flags=0, **k):
        return fd.fd_plan(*a, flags=flags, num_sms=152, **k).info
    # 32K-token decodes: one wave on 152 SMs.  By default only groups of 8 or more
    # share; a cap in the flags opens it to smaller groups.
    assert info(1, 32, 8, 128, [32768], 8, "f16")["combiners"] == 1            # G = 4
    assert info(1, 32, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_COMBINERS[8])["combiners"] == 4
    assert info(1, 64, 8, 128, [131072], 8, "f16", chunks=4,
                flags=fd.FD_PLAN_NO_CLUSTER)["combiners"] == 8                  # G = 8
    g16 = info(1, 128, 8, 128, [32768], 8, "f16")
    assert g16["path"] == 1 and g16["ctas"] == 256 and g16["combiners"] == 8   # G = 16
    g16 = info(1, 128, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_TCGEN05)
    assert g16["path"] == 3 and g16["ctas"] <= 152 and g16["combiners"] == 8   # tcgen05
    assert info(1, 8, 8, 64, [4096], 32, "f16", flags=fd.FD_PLAN_COMBINERS[16])["combiners"] == 1
    # The flags cap it; FD_PLAN_SINGLE_COMBINER is the ablation.
    for n in (1, 2, 4, 8, 16):
        want = min(n, 16)
        assert info(1, 128, 8, 128, [32768], 8, "f16",
                    flags=fd.FD_PLAN_TCGEN05 | fd.FD_PLAN_COMBINERS[n])["combiners"] == want
    # With fewer combiners each one's records outgrow the 96 KB mma.sync ring, and the
    # chunks of a segment merge in clusters first: then the last arriver combines alone.
    g16 = info(1, 128, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_COMBINERS[2])
    assert g16["records_per_segment"] == 1 and g16["combiners"] == 1
    assert info(1, 64, 8, 128, [32768], 8, "f16",
                flags=fd.FD_PLAN_SINGLE_COMBINER)["combiners"] == 1
    # Never more combiners than partials: W = 2 literal partials, G = 16.
    assert info(1, 128, 8, 128, [4096], 2, "bf16", flags=fd.FD_PLAN_LITERAL_W)["combiners"] == 2
    # Several waves (B = 64 x 16 segments = 8192 CTAs), the other launch modes and
    # clusters: the last arriver combines alone.
    assert info(64, 32, 8, 128, [8192] * 64, 16, "bf16", flags=fd.FD_PLAN_LITERAL_W)["combiners"] == 1
    for flags in (fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_WAITS, fd.FD_PLAN_CLUSTER,
                  fd.FD_PLAN_CLUSTER_COMBINE):
        assert info(1, 64, 8, 128, [32768], 8, "f16", flags=flags)["combiners"] == 1, hex(flags)
    # 128K tokens, G = 8: the 8 combiners read one head's 32 records each, which fit in
    # one pass, so the chunks need no cluster merge; with one combiner they do.
    c3 = info(1, 64, 8, 128, [131072], 8, "f16")
    assert c3["records_per_segment"] == 4 and c3["combiners"] == 8
    c3 = info(1, 64, 8, 128, [131072], 8, "f16", flags=fd.FD_PLAN_SINGLE_COMBINER)
    assert c3["records_per_segment"] == 1 and c3["combiners"] == 1


def test_drop_arrival_hook_rules():
    """FD_PLAN_TEST_DROP_ARRIVAL: a fused one-launch plan only, not with the other hooks."""
    ok = fd.fd_plan(1, 64, 8, 128, [32768], 8, "f16", flags=fd.FD_PLAN_TEST_DROP_ARRIVAL,
                    num_sms=152)
    assert ok.info["combiners"] == 8
    for other in (fd.FD_PLAN_WAITS, fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_CLUSTER_COMBINE,
                  fd.FD_PLAN_TEST_SKIP_TILE, fd.FD_PLAN_WAITS | fd.FD_PLAN_TEST_DROP_FLAG):
        assert _raw_plan(1, 64, 8, 128, [32768], [8],
                         flags=fd.FD_PLAN_TEST_DROP_ARRIVAL | other) == fd.FD_ERR_INVALID, hex(other)


def test_shallow_ring_plan_rule():
    """Three CTAs per SM with 64 KB rings for many short CTAs on the fused mma.sync path
    (G = 4 or 8, more CTAs than two per SM, <= 512 KB of K/V per CTA); two otherwise."""
    def cps(*a, flags=0, **k):
        return fd.fd_plan(*a, flags=flags, num_sms=152, **k).info["ctas_per_sm"]
    lw = fd.FD_PLAN_LITERAL_W
    # 64 sequences of 8K tokens, bf16: W = 16 and 8 (512 / 1024-token CTAs) shallow,
    # W <= 4 (2048 tokens and more) not.
    for W, want in ((16, 3), (8, 3), (4, 2), (2, 2), (1, 2)):
        assert cps(64, 32, 8, 128, [8192] * 64, W, "bf16", flags=lw) == want, W
    assert cps(64, 64, 8, 128, [8192] * 64, 16, "bf16", flags=lw) == 3          # G = 8
    assert cps(64, 128, 8, 128, [8192] * 64, 16, "bf16", flags=lw) == 2         # G = 16
    assert cps(64, 16, 8, 128, [8192] * 64, 16, "bf16", flags=lw) == 2          # G = 2: CUDA cores
    assert cps(64, 32, 8, 128, [8192] * 64, 16, "f16_e4m3kv", flags=lw) == 2    # FP8 path
    assert cps(64, 32, 8, 128, [8192] * 64, 16, "bf16", flags=lw | fd.FD_PLAN_TCGEN05) == 1
    for other in (fd.FD_PLAN_DEEP_RING, fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_CLUSTER_COMBINE):
        assert cps(64, 32, 8, 128, [8192] * 64, 16, "bf16", flags=lw | other) in (1, 2), hex(other)
    # One-wave plans keep two CTAs per SM.
    assert cps(1, 32, 8, 128, [32768], 8, "f16") == 2
    assert cps(16, 32, 8, 128, [4096] * 16, 2, "f16") == 2
