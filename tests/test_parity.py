"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (fp16/bf16 inputs, fp32 accumulation): max |out - oracle| <= 2e-3
and max |lse - oracle| <= 1e-4, element by element.  -inf lse (empty
sequences) must match exactly and their outputs must be exactly zero.

The five decode cases are held to the plain 2e-3.  Other shapes (short
sequences whose outputs are single V rows of magnitude ~1-4) may add the
output type's own rounding where that alone can reach 2e-3: an output stored
in bf16 is rounded by up to 2^-9 |x|, which exceeds 2e-3 once |x| >= 0.5; an
fp16 output by up to 2^-12 |x|, which reaches 2e-3 only for |x| >= 4.  So
bf16 outputs get half an ulp on top of 2e-3, fp16 outputs only where
|reference| >= 4, whatever the accumulation precision.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-3
LSE_TOL = 1e-4


@pytest.fixture(scope="module")
def fd():
    import split_kv_flash_decode_gb300 as fd_mod
    from split_kv_flash_decode_gb300 import build
    build.build()
    return fd_mod


def to_torch(x, dtype, device="cuda"):
    import torch
    if x.dtype == np.uint8 or dtype in ("f16", "f16_e4m3kv"):   # uint8 = FP8 E4M3 codes
        t = torch.from_numpy(np.ascontiguousarray(x))
    else:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def plan_dtype(p):
    return "f16_e4m3kv" if p.kv_type == "e4m3" else p.dtype


def reference(p):
    return oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype,
                                   kv_dtype=p.kv_dtype or None)


def out_to_f64(t):
    import torch
    return t.to(torch.float64).cpu().numpy()


def run_gpu(fd, p, chunks=0, flags=0, repeat=1):
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, plan_dtype(p),
                     flags=flags | (fd.FD_PLAN_LITERAL_W if p.literal_w else 0), chunks=chunks)
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    outs = []
    for _ in range(repeat):
        out, lse = dec(q, k, v)
        outs.append((out_to_f64(out), lse.cpu().numpy().astype(np.float64)))
    assert dec.status() == fd.FD_OK
    ws = dec.workspace.cpu().numpy()
    counters = ws[256:256 + 4 * p.B * p.Hkv].view(np.uint32)
    assert not counters.any(), "arrival counters must be back at zero"
    flag_off = 256 + -(-4 * p.B * p.Hkv // 256) * 256
    flags = ws[flag_off:flag_off + 4 * dec.info["ctas"]].view(np.uint32)
    assert not flags.any(), "ready flags must be back at zero"
    return outs if repeat > 1 else outs[0], dec


def half_ulp(x, dtype):
    """Rounding allowance of the 16-bit output type at |x|: half its spacing for
    bf16 (8 significant bits); for fp16 half its spacing only where |x| >= 4, the
    magnitude from which that alone can reach 2e-3, and zero below."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    if dtype == "f16":
        return np.where(ax >= 4.0, np.spacing(ax.astype(np.float16)).astype(np.float64) / 2, 0.0)
    e = np.floor(np.log2(np.maximum(ax, np.finfo(np.float32).tiny)))
    return np.exp2(e - 7) / 2


def check(out, lse, ref_out, ref_lse, heads=None, dtype=None):
    """Element-wise parity.  dtype=None: plain 2e-3; else 2e-3 + half an ulp of dtype."""
    if heads is not None:
        idx = tuple(np.array(heads).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(out[empty] == 0.0)
    full = ~empty
    diff = np.abs(out[full] - ref_out[full])
    bound = OUT_TOL if dtype is None else OUT_TOL + half_ulp(ref_out[full], dtype)
    excess = (diff - bound).max(initial=-1.0)
    err_o = diff.max(initial=0.0)
    err_l = np.abs(lse[full] - ref_lse[full]).max(initial=0.0)
    assert excess <= 0.0, f"max |out err| {err_o:.3e} exceeds its bound by {excess:.3e}"
    assert err_l <= LSE_TOL, f"max |lse err| {err_l:.3e}"
    return err_o, err_l


# ---------------------------------------------------------------------------
# The five decode cases at full size.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["mha8_d64_L4k_W4", "gqa4_d128_L32k_W8", "gqa8_d128_L128k_W8_spiky"])
def test_case_full(fd, name):
    p = workloads.CASES[name]()
    (out, lse), _ = run_gpu(fd, p)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out, lse, ref_out, ref_lse)


def test_spiky_128k_bf16_full(fd):
    """The wide-logit case in bf16 (not one of the five cases).  A few x20 keys dominate,
    so outputs reach |x| in [2, 4), where storing a bf16 result alone rounds by up to
    2^-7 = 7.8e-3: the bound is 2e-3 plus that half ulp.  P and its row sums use the
    same rounded weights, so no error beyond the output's own rounding appears."""
    p = workloads.gqa8_d128_L128k_W8_spiky(dtype="bf16")
    (out, lse), _ = run_gpu(fd, p)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out, lse, ref_out, ref_lse, dtype="bf16")


def test_ragged16_full(fd):
    p = workloads.ragged16_gqa4_d128()
    (out, lse), _ = run_gpu(fd, p)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out, lse, ref_out, ref_lse)


def test_batch64_bf16_w_sweep_deterministic(fd):
    p1 = workloads.batch64_gqa4_d128_L8k_bf16(W=1)
    ref_out, ref_lse = oracle.decode_reference(p1.q, p1.k, p1.v, p1.seqlens, p1.dtype)
    for W in workloads.W_SWEEP:
        p = workloads.batch64_gqa4_d128_L8k_bf16(W=W)
        runs, dec = run_gpu(fd, p, repeat=20 if W == 16 else 2)
        assert dec.info["chunks"] == 1 and dec.info["ctas"] == 64 * 8 * W
        out0, lse0 = runs[0]
        for out, lse in runs[1:]:
            assert np.array_equal(out, out0) and np.array_equal(lse, lse0), "not bitwise deterministic"
        check(out0, lse0, ref_out, ref_lse)


@pytest.mark.parametrize("dtype,G,d", [("bf16", 4, 128), ("f16", 8, 128), ("bf16", 4, 64)])
def test_shallow_ring_matches_deep_ring(fd, dtype, G, d):
    """Many short CTAs: the three-per-SM build (64 KB rings) agrees with the oracle and,
    bit for bit, with the two-per-SM build (FD_PLAN_DEEP_RING): the ring depth changes
    the schedule, not the arithmetic."""
    rs = np.random.default_rng(140 + G + d)
    lens = [int(x) for x in rs.integers(1, 3000, size=40)] + [0, 1, 64, 4096]
    p = workloads.make_problem("shallow", len(lens), 8 * G, 8, d, lens, 8, dtype, seed=141 + G + d)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    (o1, l1), dec = run_gpu(fd, p)
    assert dec.info["ctas_per_sm"] == 3 and dec.info["ctas"] > 2 * 152
    check(o1, l1, ref_out, ref_lse, dtype=dtype)
    (o2, l2), dec2 = run_gpu(fd, p, flags=fd.FD_PLAN_DEEP_RING)
    assert dec2.info["ctas_per_sm"] == 2 and dec2.info["chunks"] == dec.info["chunks"]
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("page_size", [16, 64])
def test_shallow_ring_paged(fd, page_size):
    """Many short CTAs over a paged cache: the three-per-SM build against the oracle and,
    bit for bit, against the two-per-SM build."""
    rs = np.random.default_rng(150 + page_size)
    lens = [int(x) for x in rs.integers(1, 2500, size=44)]
    p = workloads.make_problem("shallow_paged", len(lens), 32, 8, 128, lens, 8, "bf16",
                               seed=151 + page_size)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    o1, l1, dec, _ = run_paged(fd, p, page_size)
    assert dec.info["ctas_per_sm"] == 3
    check(o1, l1, ref_out, ref_lse, dtype=p.dtype)
    o2, l2, dec2, _ = run_paged(fd, p, page_size, flags=fd.FD_PLAN_DEEP_RING)
    assert dec2.info["ctas_per_sm"] == 2
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_shallow_ring_batch64_w16(fd):
    """The default bench case on the shallow ring: bitwise equal to the deep ring."""
    p = workloads.batch64_gqa4_d128_L8k_bf16(W=16)
    (o1, l1), dec = run_gpu(fd, p)
    assert dec.info["ctas_per_sm"] == 3
    (o2, l2), _ = run_gpu(fd, p, flags=fd.FD_PLAN_DEEP_RING)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------------------
# Edge shapes: tile boundaries, W beyond L, every G and d, both dtypes.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_edge_lengths(fd, dtype, d, G):
    Hkv = 2
    lens = [1, 2, 31, 32, 33, 63, 64, 65, 97, 1000]
    W = [1, 3, 31, 1, 40, 2, 64, 70, 5, 7]
    p = workloads.make_problem("edge", len(lens), Hkv * G, Hkv, d, lens, W, dtype, seed=7 + G + d)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (0, 1, 3):
        (out, lse), _ = run_gpu(fd, p, chunks=chunks)
        check(out, lse, ref_out, ref_lse, dtype=dtype)


@pytest.mark.parametrize("G", [4, 8])
def test_forced_ffma_path(fd, G):
    """The CUDA-core consumers stay correct for the groups the tensor-core path serves."""
    p = workloads.make_problem("ffma", 2, 8 * G, 8, 128, [3000, 77], [3, 5], "f16", seed=20 + G)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    (out, lse), dec = run_gpu(fd, p, flags=fd.FD_PLAN_FFMA)
    assert dec.info["path"] == 0
    check(out, lse, ref_out, ref_lse, dtype=p.dtype)


@pytest.mark.parametrize("dtype,d", [("f16", 128), ("bf16", 64), ("bf16", 128)])
def test_gqa16_tensor_core_path(fd, dtype, d):
    """G = 16 query heads per KV head: two mma.sync N tiles per KV tile by default,
    tcgen05 at d = 128 with FD_PLAN_TCGEN05."""
    p = workloads.make_problem("gqa16", 3, 128, 8, d, [9000, 1, 2049], [4, 1, 3], dtype,
                               seed=60 + d)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for tc in ((False, True) if d == 128 else (False,)):
        for flags in (0, fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_WAITS):
            (out, lse), dec = run_gpu(fd, p, flags=flags | (fd.FD_PLAN_TCGEN05 if tc else 0))
            assert dec.info["path"] == (3 if tc else 1) and dec.info["G"] == 16
            check(out, lse, ref_out, ref_lse, dtype=p.dtype)


# ---------------------------------------------------------------------------
# tcgen05 consumers (FD_PLAN_TCGEN05): 128-token tiles, accumulators in tensor memory.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [4, 8, 16])
def test_tcgen05_edge_lengths(fd, dtype, G):
    """Tile boundaries of the 128-token tiles, W beyond L, empty sequences, C in {auto, 1, 3}."""
    Hkv = 2
    lens = [1, 2, 127, 128, 129, 255, 256, 257, 0, 1000, 3001]
    W = [1, 3, 1, 2, 40, 1, 2, 3, 2, 7, 4]
    p = workloads.make_problem("tc_edge", len(lens), Hkv * G, Hkv, 128, lens, W, dtype,
                               seed=100 + G)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (0, 1, 3):
        (out, lse), dec = run_gpu(fd, p, chunks=chunks, flags=fd.FD_PLAN_TCGEN05)
        assert dec.info["path"] == 3
        check(out, lse, ref_out, ref_lse, dtype=dtype)


@pytest.mark.parametrize("dtype,G", [("f16", 4), ("bf16", 8), ("f16", 16)])
def test_tcgen05_variants(fd, dtype, G):
    """Fused (bitwise across runs), two launches (bitwise equal to fused), in-cluster
    segment merge, fine-grained waits, and paged caches, all against the oracle."""
    p = workloads.make_problem("tc_var", 3, 8 * G, 8, 128, [9000, 17, 4096], [4, 2, 8], dtype,
                               seed=110 + G)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    runs, _ = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05, repeat=3)
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
    check(*runs[0], ref_out, ref_lse, dtype=dtype)
    (o2, l2), _ = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05 | fd.FD_PLAN_TWO_LAUNCH)
    assert np.array_equal(o2, runs[0][0]) and np.array_equal(l2, runs[0][1])
    for flags in (fd.FD_PLAN_CLUSTER, fd.FD_PLAN_WAITS, fd.FD_PLAN_NO_PDL):
        (o3, l3), _ = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05 | flags)
        check(o3, l3, ref_out, ref_lse, dtype=dtype)
    for page_size in (16, 128, 256):
        out, lse, dec, _ = run_paged(fd, p, page_size, flags=fd.FD_PLAN_TCGEN05)
        assert dec.info["path"] == 3
        check(out, lse, ref_out, ref_lse, dtype=dtype)


@pytest.mark.parametrize("name", ["gqa4_d128_L32k_W8", "gqa8_d128_L128k_W8_spiky",
                                  "ragged16_gqa4_d128", "gqa16_d128_L32k_W8"])
def test_tcgen05_full_cases(fd, name):
    p = (workloads.CASES.get(name) or workloads.EXTRA[name])()
    (out, lse), dec = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05)
    assert dec.info["path"] == 3
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out, lse, ref_out, ref_lse)


def test_tcgen05_batch64_bf16_w16(fd):
    """The largest decode case (2.15 GB of K/V) on tcgen05, W = 16: against the oracle,
    and bitwise across repeats."""
    p = workloads.batch64_gqa4_d128_L8k_bf16(W=16)
    runs, dec = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05, repeat=3)
    assert dec.info["path"] == 3 and dec.info["ctas"] == 64 * 8 * 16
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(*runs[0], ref_out, ref_lse)


def test_tcgen05_closed_forms(fd):
    """Equal V rows return that row; q = 0 gives the mean of V and lse = ln L."""
    rs = np.random.default_rng(120)
    L, Hkv, G, d = 3000, 2, 8, 128
    p = workloads.make_problem("tc_closed", 1, Hkv * G, Hkv, d, [L], 4, "f16", seed=120)
    row = rs.standard_normal((Hkv, d)).astype(np.float16)
    p.v[:] = row[None]
    (out, lse), _ = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05)
    for h in range(Hkv * G):
        assert np.abs(out[0, h] - row[h // G].astype(np.float64)).max() <= 1e-3
    p.q[:] = 0
    p.v[:] = rs.standard_normal(p.v.shape).astype(np.float16)
    (out, lse), _ = run_gpu(fd, p, flags=fd.FD_PLAN_TCGEN05)
    mean = p.v.astype(np.float64).mean(axis=0)
    for h in range(Hkv * G):
        assert np.abs(out[0, h] - mean[h // G]).max() <= OUT_TOL
    assert np.abs(lse - np.log(L)).max() <= LSE_TOL


# ---------------------------------------------------------------------------
# Combine inside a thread-block cluster per (sequence, KV head) (FD_PLAN_CLUSTER_COMBINE).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,G,d,extra", [("f16", 1, 64, 0), ("bf16", 2, 128, 0),
                                             ("f16", 4, 128, 0), ("bf16", 8, 64, 0),
                                             ("f16", 16, 128, 0), ("bf16", 4, 128, "tcgen05"),
                                             ("f16", 16, 128, "tcgen05"), ("f16", 8, 128, "ffma")])
def test_cluster_combine(fd, dtype, G, d, extra):
    """Edge lengths, empty sequences, W beyond L and C in {auto, 1, 4}: against the oracle,
    and bitwise across runs (the combine order inside the cluster is fixed)."""
    flag = fd.FD_PLAN_CLUSTER_COMBINE | {0: 0, "tcgen05": fd.FD_PLAN_TCGEN05,
                                         "ffma": fd.FD_PLAN_FFMA}[extra]
    lens = [1, 2, 127, 128, 129, 0, 1000, 3001, 9000]
    p = workloads.make_problem("cc", len(lens), 2 * G, 2, d, lens, 4, dtype, seed=130 + G + d)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (0, 1, 4):
        runs, dec = run_gpu(fd, p, chunks=chunks, flags=flag, repeat=2)
        assert dec.info["combine_cluster"] == 4 * dec.info["chunks"]
        assert np.array_equal(runs[0][0], runs[1][0]) and np.array_equal(runs[0][1], runs[1][1])
        check(*runs[0], ref_out, ref_lse, dtype=dtype)


@pytest.mark.parametrize("name", ["gqa4_d128_L32k_W8", "gqa8_d128_L128k_W8_spiky",
                                  "gqa16_d128_L32k_W8", "mha8_d64_L4k_W4"])
@pytest.mark.parametrize("tcgen05", [False, True])
def test_cluster_combine_full_cases(fd, name, tcgen05):
    p = (workloads.CASES.get(name) or workloads.EXTRA[name])()
    if tcgen05 and p.Hq // p.Hkv < 4:
        pytest.skip("tcgen05 consumers need G >= 4")
    flags = fd.FD_PLAN_CLUSTER_COMBINE | (fd.FD_PLAN_TCGEN05 if tcgen05 else 0)
    (out, lse), dec = run_gpu(fd, p, flags=flags)
    assert dec.info["combine_cluster"] >= 2
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out, lse, ref_out, ref_lse)


def test_cluster_combine_batch64_w_sweep(fd):
    """The W sweep of the bf16 batch with clusters of W CTAs: against the oracle, and
    bitwise across repeats."""
    p1 = workloads.batch64_gqa4_d128_L8k_bf16(W=1)
    ref_out, ref_lse = oracle.decode_reference(p1.q, p1.k, p1.v, p1.seqlens, p1.dtype)
    for W in (2, 16):
        p = workloads.batch64_gqa4_d128_L8k_bf16(W=W)
        runs, dec = run_gpu(fd, p, flags=fd.FD_PLAN_CLUSTER_COMBINE, repeat=3)
        assert dec.info["combine_cluster"] == W
        for o, l in runs[1:]:
            assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
        check(*runs[0], ref_out, ref_lse)


def test_cluster_combine_fp8_and_paged(fd):
    base = workloads.make_problem("cc8", 3, 64, 8, 128, [7000, 0, 2049], 4, "f16", seed=140)
    p = workloads.with_e4m3_kv(base)
    ref_out, ref_lse = reference(p)
    (out, lse), dec = run_gpu(fd, p, flags=fd.FD_PLAN_CLUSTER_COMBINE)
    assert dec.info["path"] == 2
    check(out, lse, ref_out, ref_lse, dtype="f16")
    q = workloads.make_problem("ccp", 3, 32, 8, 128, [7000, 33, 2049], 4, "bf16", seed=141)
    ref_out, ref_lse = oracle.decode_reference(q.q, q.k, q.v, q.seqlens, q.dtype)
    for flags in (fd.FD_PLAN_CLUSTER_COMBINE, fd.FD_PLAN_CLUSTER_COMBINE | fd.FD_PLAN_TCGEN05):
        out, lse, dec, _ = run_paged(fd, q, 64, flags=flags)
        check(out, lse, ref_out, ref_lse, dtype="bf16")


def test_ragged_with_empty_sequences(fd):
    lens = [0, 700, 0, 1, 4096, 0]
    p = workloads.make_problem("ragged_empty", 6, 16, 4, 128, lens, [1, 3, 5, 2, 4, 1], "f16", seed=11)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (0, 2):
        (out, lse), _ = run_gpu(fd, p, chunks=chunks)
        check(out, lse, ref_out, ref_lse, dtype=p.dtype)


def test_all_sequences_empty(fd):
    p = workloads.make_problem("all_empty", 3, 8, 8, 64, [0, 0, 0], 2, "bf16", seed=12)
    (out, lse), _ = run_gpu(fd, p)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_chunk_counts_agree(fd):
    p = workloads.make_problem("chunks", 2, 32, 8, 128, [5000, 3001], [3, 2], "f16", seed=13)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (1, 2, 5, 16, 100):
        (out, lse), _ = run_gpu(fd, p, chunks=chunks)
        check(out, lse, ref_out, ref_lse, dtype=p.dtype)


def test_closed_forms_on_gpu(fd):
    """Equal V rows return that row; q = 0 returns the mean of V with lse = ln L."""
    rs = np.random.default_rng(14)
    L, Hkv, G, d = 3000, 2, 4, 128
    p = workloads.make_problem("closed", 1, Hkv * G, Hkv, d, [L], 4, "f16", seed=14)
    row = rs.standard_normal((Hkv, d)).astype(np.float16)
    p.v[:] = row[None]
    (out, lse), _ = run_gpu(fd, p)
    for h in range(Hkv * G):
        assert np.abs(out[0, h] - row[h // G].astype(np.float64)).max() <= 1e-3
    p.q[:] = 0
    p.v[:] = rs.standard_normal(p.v.shape).astype(np.float16)
    (out, lse), _ = run_gpu(fd, p)
    mean = p.v.astype(np.float64).mean(axis=0)
    for h in range(Hkv * G):
        assert np.abs(out[0, h] - mean[h // G]).max() <= OUT_TOL
    assert np.abs(lse - np.log(L)).max() <= LSE_TOL


def test_two_launch_matches_fused(fd):
    p = workloads.make_problem("two_launch", 3, 32, 8, 128, [9000, 17, 4096], [4, 2, 8], "bf16", seed=15)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    (o1, l1), _ = run_gpu(fd, p)
    (o2, l2), _ = run_gpu(fd, p, flags=fd.FD_PLAN_TWO_LAUNCH)
    check(o2, l2, ref_out, ref_lse, dtype=p.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("dtype,G,d", [("f16", 4, 128), ("bf16", 8, 128), ("f16", 16, 128),
                                       ("bf16", 1, 64), ("f16", 2, 128), ("bf16", 16, 64)])
def test_cluster_segment_merge(fd, dtype, G, d):
    """Chunks merged per segment inside a cluster (forced) agree with the oracle, with
    one record per chunk (FD_PLAN_NO_CLUSTER), and between runs bitwise."""
    p = workloads.make_problem("cluster", 3, 4 * G, 4, d, [9000, 1, 2500], [4, 1, 3], dtype,
                               seed=80 + G + d)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (2, 3, 8):
        runs, dec = run_gpu(fd, p, chunks=chunks, repeat=3, flags=fd.FD_PLAN_CLUSTER)
        assert dec.info["chunks"] == chunks and dec.info["records_per_segment"] == 1
        for o, l in runs[1:]:
            assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
        check(*runs[0], ref_out, ref_lse, dtype=p.dtype)
        (o2, l2), dec2 = run_gpu(fd, p, chunks=chunks, flags=fd.FD_PLAN_NO_CLUSTER)
        assert dec2.info["records_per_segment"] == chunks
        check(o2, l2, ref_out, ref_lse, dtype=p.dtype)
        (o3, l3), _ = run_gpu(fd, p, chunks=chunks,
                              flags=fd.FD_PLAN_TWO_LAUNCH | fd.FD_PLAN_CLUSTER)
        assert np.array_equal(o3, runs[0][0]) and np.array_equal(l3, runs[0][1])


def test_pdl_off_matches_pdl_on(fd):
    """Programmatic dependent launch changes scheduling only, never the numbers."""
    p = workloads.make_problem("pdl", 2, 32, 8, 128, [6000, 999], [4, 3], "f16", seed=18)
    (o1, l1), _ = run_gpu(fd, p, repeat=1)
    (o2, l2), _ = run_gpu(fd, p, flags=fd.FD_PLAN_NO_PDL)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("dtype,G,d", [("f16", 4, 128), ("bf16", 8, 128), ("f16", 1, 64),
                                       ("bf16", 4, 64)])
def test_fine_grained_waits_variant(fd, dtype, G, d):
    """Slot 0 of each (sequence, KV head) combines the partials as their flags arrive."""
    p = workloads.make_problem("waits", 3, 8 * G, 8, d, [20000, 0, 3001], [4, 2, 3], dtype,
                               seed=30 + G + d)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (0, 1):
        (out, lse), dec = run_gpu(fd, p, flags=fd.FD_PLAN_WAITS, chunks=chunks)
        check(out, lse, ref_out, ref_lse, dtype=p.dtype)


def test_fine_grained_waits_full_32k(fd):
    p = workloads.gqa4_d128_L32k_W8()
    (out, lse), dec = run_gpu(fd, p, flags=fd.FD_PLAN_WAITS)
    assert dec.info["ctas"] == 256
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out, lse, ref_out, ref_lse)


def test_fine_grained_waits_timeout_is_reported(fd):
    """A flag that nothing sets: the bounded wait gives up, the status word says so,
    the other (sequence, KV head) pairs are still correct and the context stays usable."""
    import torch
    p = workloads.make_problem("timeout", 2, 16, 4, 128, [5000, 700], [4, 2], "f16", seed=40)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype,
                     flags=fd.FD_PLAN_WAITS | fd.FD_PLAN_TEST_DROP_FLAG)
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((p.B, p.Hq), float("nan"), dtype=torch.float32, device="cuda")
    dec(q, k, v, out, lse)
    assert dec.status() == fd.FD_ERR_TIMEOUT
    o, l = out_to_f64(out), lse.cpu().numpy().astype(np.float64)
    G = p.Hq // p.Hkv
    assert np.isnan(o[0, :G]).all() and np.isnan(l[0, :G]).all()   # the starved pair: untouched
    keep = np.ones((p.B, p.Hq), dtype=bool)
    keep[0, :G] = False
    assert np.abs(o[keep] - ref_out[keep]).max() <= OUT_TOL
    assert np.abs(l[keep] - ref_lse[keep]).max() <= LSE_TOL
    # Same context, clean workspace, no dropped flag: a normal decode.
    (out2, lse2), _ = run_gpu(fd, p, flags=fd.FD_PLAN_WAITS)
    check(out2, lse2, ref_out, ref_lse, dtype=p.dtype)


@pytest.mark.parametrize("G,flags", [(4, 0), (4, "two_launch"), (8, "cluster"), (1, 0),
                                     (8, "tcgen05"), (16, "tcgen05_cluster"),
                                     (4, "cluster_combine"), (4, "single_combiner")])
def test_pipeline_wait_timeout_leaves_workspace_clean(fd, G, flags):
    """A tile that is never loaded (test hook): the consumers' bounded wait gives up,
    the status word says so, the CTA still publishes an (empty) partial and arrives, so
    every counter returns to zero; the other (sequence, KV head) pairs are correct, and
    the next decode on the same workspace, without re-initialising it, is correct."""
    import torch
    flag = {0: 0, "two_launch": fd.FD_PLAN_TWO_LAUNCH, "cluster": fd.FD_PLAN_CLUSTER,
            "tcgen05": fd.FD_PLAN_TCGEN05,
            "tcgen05_cluster": fd.FD_PLAN_TCGEN05 | fd.FD_PLAN_CLUSTER,
            "cluster_combine": fd.FD_PLAN_CLUSTER_COMBINE,
            "single_combiner": fd.FD_PLAN_SINGLE_COMBINER}[flags]
    W = 4 if flags == "cluster_combine" else [4, 2]      # one W for every sequence there
    p = workloads.make_problem("skip", 2, 4 * G, 4, 128, [5000, 700], W, "f16", seed=42 + G)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype,
                     flags=flag | fd.FD_PLAN_TEST_SKIP_TILE)
    lo, hi = dec.plan.range(0, 0)
    assert hi - lo > 128, "slot 0 of sequence 0 must span two tiles for the hook to act"
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((p.B, p.Hq), float("nan"), dtype=torch.float32, device="cuda")
    dec(q, k, v, out, lse)
    assert dec.status() == fd.FD_ERR_TIMEOUT
    ws = dec.workspace.cpu().numpy()
    assert not ws[256:256 + 4 * p.B * p.Hkv].view(np.uint32).any(), "counters not back at zero"
    o, l = out_to_f64(out), lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all() and np.isfinite(l).all(), "every pair was combined and written"
    keep = np.ones((p.B, p.Hq), dtype=bool)
    keep[0, :G] = False                     # (sequence 0, KV head 0) lacks the starved partial
    assert np.abs(o[keep] - ref_out[keep]).max() <= OUT_TOL
    assert np.abs(l[keep] - ref_lse[keep]).max() <= LSE_TOL
    clean = fd.fd_plan(p.B, p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype, flags=flag)
    assert clean.workspace_bytes == dec.plan.workspace_bytes
    out2 = torch.empty_like(q)
    lse2 = torch.empty_like(lse)
    fd.fd_decode(clean, q, k, v, out2, lse2, dec.workspace)
    assert fd.fd_workspace_status(clean, dec.workspace) == fd.FD_OK
    check(out_to_f64(out2), lse2.cpu().numpy().astype(np.float64), ref_out, ref_lse, dtype=p.dtype)


# Shapes for the shared combine: (dtype, G, d, B, Hkv, seqlens, W, kind, combiners
# wanted); groups below 8 share only under a cap in the flags (kind "cap").  Ragged partial counts give some sequences fewer combiners than others
# (or none, W = 1 literal); Hkv = 1 with 300 literal partials sends each combiner's
# head to the combine that reads the records from L2; 8 heads of 32 records per
# combiner need two passes through the 96 KB ring.
SHARED_COMBINE_CASES = {
    "gqa4_f16": ("f16", 4, 128, 3, 8, [9000, 17, 4096], [4, 2, 8], "cap", 4),
    "gqa8_bf16_literal": ("bf16", 8, 128, 3, 8, [9000, 300, 4096], [4, 1, 3], "literal", 4),
    "gqa16_mma": ("f16", 16, 128, 2, 4, [20000, 3000], [8, 3], "", 8),
    "gqa16_tcgen05": ("f16", 16, 128, 2, 4, [20000, 3000], [8, 3], "tcgen05", 8),
    "gqa16_two_passes": ("bf16", 16, 128, 1, 2, [40000], [8], "two_passes", 2),
    "gqa4_from_l2": ("f16", 4, 128, 1, 1, [300 * 64], [300], "literal_cap", 4),
    "gqa2_d64_ffma": ("bf16", 2, 64, 2, 8, [5000, 100], [4, 4], "cap", 2),
    "gqa8_e4m3": ("e4m3", 8, 128, 3, 8, [7000, 0, 2049], [4, 2, 3], "", 8),
}


@pytest.mark.parametrize("case", list(SHARED_COMBINE_CASES))
def test_shared_combine_matches_single_combiner(fd, case):
    """The last arrivals of a pair share its combine by query heads: bit-identical to
    the last arriver combining alone over the same records, and both agree with the
    oracle.  (No cluster merge: a single combiner's plan could otherwise merge chunks
    per segment, which changes the order of the sums.)"""
    dtype, G, d, B, Hkv, seqlens, W, kind, want = SHARED_COMBINE_CASES[case]
    base = workloads.make_problem("shared_combine", B, G * Hkv, Hkv, d, seqlens, W,
                                  "f16" if dtype == "e4m3" else dtype, seed=130 + len(case))
    p = workloads.with_e4m3_kv(base) if dtype == "e4m3" else base
    flags, chunks = fd.FD_PLAN_NO_CLUSTER, 0
    if kind.startswith("literal"):
        flags |= fd.FD_PLAN_LITERAL_W
    if kind.endswith("cap"):
        flags |= fd.FD_PLAN_COMBINERS[16]
    elif kind == "two_passes":
        flags, chunks = flags | fd.FD_PLAN_MMA_SYNC | fd.FD_PLAN_COMBINERS[2], 4
    elif kind == "tcgen05":
        flags |= fd.FD_PLAN_TCGEN05
    ref_out, ref_lse = reference(p)
    (o1, l1), dec = run_gpu(fd, p, flags=flags, chunks=chunks)
    assert dec.info["combiners"] == want
    check(o1, l1, ref_out, ref_lse, dtype=p.dtype)
    single = (flags & ~fd.FD_PLAN_COMBINERS_MASK) | fd.FD_PLAN_SINGLE_COMBINER
    (o2, l2), dec2 = run_gpu(fd, p, flags=single, chunks=chunks)
    assert dec2.info["combiners"] == 1
    assert dec2.info["records_per_segment"] == dec.info["records_per_segment"]
    check(o2, l2, ref_out, ref_lse, dtype=p.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_shared_combine_wait_runs_out(fd):
    """A partial that never arrives (test hook): the pair's combiners wait for the last
    arrival, give up after their bound (~4 s) and report FD_ERR_TIMEOUT; that pair's
    out/lse stay untouched, every other pair is correct, and after fd_workspace_init
    the next decode on the same workspace is correct."""
    import torch
    p = workloads.make_problem("drop_arrival", 2, 32, 4, 128, [5000, 700], [4, 2], "f16", seed=77)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype, flags=fd.FD_PLAN_TEST_DROP_ARRIVAL)
    assert dec.info["combiners"] > 1 and dec.plan.range(0, 1)[1] > dec.plan.range(0, 1)[0]
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((p.B, p.Hq), float("nan"), dtype=torch.float32, device="cuda")
    dec(q, k, v, out, lse)
    assert dec.status() == fd.FD_ERR_TIMEOUT
    o, l = out_to_f64(out), lse.cpu().numpy().astype(np.float64)
    G = p.Hq // p.Hkv
    assert np.isnan(o[0, :G]).all() and np.isnan(l[0, :G]).all()   # the pair nobody combined
    keep = np.ones((p.B, p.Hq), dtype=bool)
    keep[0, :G] = False
    assert np.abs(o[keep] - ref_out[keep]).max() <= OUT_TOL
    assert np.abs(l[keep] - ref_lse[keep]).max() <= LSE_TOL
    clean = fd.fd_plan(p.B, p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype)
    assert clean.workspace_bytes == dec.plan.workspace_bytes
    fd.fd_workspace_init(clean, dec.workspace)
    out2, lse2 = torch.empty_like(q), torch.empty_like(lse)
    fd.fd_decode(clean, q, k, v, out2, lse2, dec.workspace)
    assert fd.fd_workspace_status(clean, dec.workspace) == fd.FD_OK
    check(out_to_f64(out2), lse2.cpu().numpy().astype(np.float64), ref_out, ref_lse, dtype=p.dtype)


def test_fine_grained_waits_needs_coresidency(fd):
    p = workloads.make_problem("big", 64, 32, 8, 128, [512] * 64, 16, "bf16", seed=41)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype,
                     flags=fd.FD_PLAN_WAITS | fd.FD_PLAN_LITERAL_W)
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    with pytest.raises(fd.FdError) as ei:
        dec(q, k, v)                       # 8192 CTAs cannot all be resident: refused
    assert ei.value.status == fd.FD_ERR_UNSUPPORTED


def run_paged(fd, p, page_size, flags=0, chunks=0):
    import torch
    kp, vp, table = workloads.to_paged(p, page_size)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, plan_dtype(p), flags=flags, chunks=chunks,
                     page_size=page_size)
    q = to_torch(p.q, p.dtype)
    out, lse = dec.decode_paged(q, to_torch(kp, p.dtype), to_torch(vp, p.dtype),
                                torch.from_numpy(table).cuda())
    assert dec.status() == fd.FD_OK
    return out_to_f64(out), lse.cpu().numpy().astype(np.float64), dec, (kp, vp, table)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype,G", [("f16", 4), ("bf16", 8), ("f16", 1)])
def test_paged_cache(fd, page_size, dtype, G):
    p = workloads.make_problem("paged", 4, 8 * G, 8, 128, [5000, 0, 33, 1031], [3, 1, 2, 4], dtype,
                               seed=50 + page_size + G)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for chunks in (0, 2):
        out, lse, dec, (kp, vp, table) = run_paged(fd, p, page_size, chunks=chunks)
        check(out, lse, ref_out, ref_lse, dtype=p.dtype)
    # the oracle over the gathered pages is the same problem
    k, v = oracle.gather_paged(kp, vp, table, p.seqlens, page_size)
    assert np.array_equal(k, p.k) and np.array_equal(v, p.v)


def test_paged_cache_full_32k_and_variants(fd):
    p = workloads.gqa4_d128_L32k_W8()
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    for flags in (0, fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_WAITS, fd.FD_PLAN_CLUSTER):
        out, lse, _, _ = run_paged(fd, p, 64, flags=flags)
        check(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("G", [4, 8, 16])
def test_fp8_e4m3_kv_cache(fd, G):
    """fp16 q over an FP8 (E4M3) cache, against the oracle on the same E4M3 values."""
    base = workloads.make_problem("fp8kv", 3, 8 * G, 8, 128, [7000, 0, 2049], [4, 2, 3], "f16",
                                  seed=70 + G)
    p = workloads.with_e4m3_kv(base)
    ref_out, ref_lse = reference(p)
    for flags in (0, fd.FD_PLAN_TWO_LAUNCH, fd.FD_PLAN_WAITS, fd.FD_PLAN_CLUSTER):
        (out, lse), dec = run_gpu(fd, p, flags=flags)
        assert dec.info["path"] == 2 and dec.info["kv_bytes"] == p.kv_bytes
        check(out, lse, ref_out, ref_lse, dtype="f16")
    for page_size, flags in ((16, 0), (128, 0), (64, fd.FD_PLAN_CLUSTER)):
        out, lse, dec, _ = run_paged(fd, p, page_size, flags=flags)
        if flags:
            assert dec.info["records_per_segment"] == 1
        check(out, lse, ref_out, ref_lse, dtype="f16")


def test_fp8_e4m3_kv_full_cases(fd):
    for make in (workloads.gqa4_d128_L32k_W8, workloads.gqa8_d128_L128k_W8_spiky):
        p = workloads.with_e4m3_kv(make())
        ref_out, ref_lse = reference(p)
        (out, lse), _ = run_gpu(fd, p)
        check(out, lse, ref_out, ref_lse)


def test_fp8_nan_codes_propagate(fd):
    """OCP E4M3 gives codes 0x7F / 0xFF no value (NaN).  The kernel widens cache bytes
    with the hardware conversion, which reads them as NaN, as the oracle does: a NaN
    key makes every output and the lse of its query heads NaN; a NaN value makes that
    dimension of their outputs NaN.  The NaN pattern must match the oracle's exactly,
    and every other element must match within the tolerances."""
    base = workloads.make_problem("fp8nan", 1, 32, 8, 128, [300], 2, "f16", seed=75)
    p = workloads.with_e4m3_kv(base)
    p.k[17, 3, 5] = 0x7F          # KV head 3 -> query heads 12..15
    p.v[200, 1, 9] = 0xFF         # KV head 1 -> query heads 4..7, dimension 9
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, "f16", kv_dtype="e4m3")
    assert np.isnan(ref_out[0, 12:16]).all() and np.isnan(ref_lse[0, 12:16]).all()
    assert np.isnan(ref_out[0, 4:8, 9]).all() and not np.isnan(ref_lse[0, 4:8]).any()
    for flags in (0, fd.FD_PLAN_TWO_LAUNCH):
        (out, lse), _ = run_gpu(fd, p, flags=flags)
        diff = np.argwhere(np.isnan(out) != np.isnan(ref_out))
        assert len(diff) == 0, (f"{len(diff)} elements differ in NaN-ness, e.g. "
                                f"{diff[:4].tolist()}; kernel NaN count {int(np.isnan(out).sum())}, "
                                f"oracle {int(np.isnan(ref_out).sum())}")
        assert np.array_equal(np.isnan(lse), np.isnan(ref_lse))
        fo, fl = ~np.isnan(ref_out), ~np.isnan(ref_lse)
        assert np.abs(out[fo] - ref_out[fo]).max() <= OUT_TOL
        assert np.abs(lse[fl] - ref_lse[fl]).max() <= LSE_TOL


def test_debug_plan_detects_counter_state(fd):
    import torch
    p = workloads.make_problem("debug", 1, 8, 8, 64, [2048], 4, "f16", seed=16)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype, flags=fd.FD_PLAN_DEBUG)
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    dec(q, k, v)                                      # clean workspace: ok
    dec.workspace[256:260] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")
    with pytest.raises(fd.FdError) as ei:
        dec(q, k, v)                                  # host check, nothing launched
    assert ei.value.status == fd.FD_ERR_STATE
    fd.fd_workspace_init(dec.plan, dec.workspace)
    out, lse = dec(q, k, v)
    ref_out, ref_lse = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    check(out_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, dtype=p.dtype)


def test_lse_optional_and_misaligned_rejected(fd):
    import torch
    p = workloads.make_problem("opt", 1, 8, 8, 64, [300], 2, "f16", seed=17)
    dec = fd.Decoder(p.Hq, p.Hkv, p.d, p.seqlens, p.W, p.dtype)
    q, k, v = (to_torch(x, p.dtype) for x in (p.q, p.k, p.v))
    out = torch.empty_like(q)
    fd.fd_decode(dec.plan, q, k, v, out, None, dec.workspace)
    ref_out, _ = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    assert np.abs(out_to_f64(out) - ref_out).max() <= OUT_TOL
    with pytest.raises(fd.FdError) as ei:
        fd.fd_decode(dec.plan, q, k, v, out.view(-1)[1:].data_ptr(), None, dec.workspace)
    assert ei.value.status == fd.FD_ERR_ALIGN
