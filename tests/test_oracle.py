"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: hand-derived closed
forms (tests/golden), pure-Python brute force that takes a different numeric
route (no max shift, exact fsum), library routines (torch SDPA, logsumexp),
invariants of softmax attention, and the associativity/commutativity of
OnlineSoftmaxCombine ("Eliminating Multi-GPU Performance Taxes" review page,
core equations and correctness check #5).  The last test plants mistakes in
the oracle and checks that these pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import fd_oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_decode.json")
TOL = 1e-12


def _ev(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"ln": math.log, "inf": math.inf}))
    return float(x)


def _arr(x):
    if isinstance(x, list):
        return np.array([_arr(e) for e in x], dtype=np.float64)
    return _ev(x)


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _rand_f64(rs, shape, scale=1.0):
    return rs.standard_normal(shape) * scale


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(diff <= tol))


# ---------------------------------------------------------------------------
# Pin checks (each returns True when the oracle passes; reused by the
# planted-mistake test below).
# ---------------------------------------------------------------------------

def check_golden():
    for c in _golden_cases():
        q, k, v = _arr(c["q"]), _arr(c["k"]), _arr(c["v"])
        out_ref, lse_ref = _arr(c["out"]), _arr(c["lse"])
        o1, l1 = oracle.decode_reference(q, k, v, c["seqlens"], dtype="f64")
        o2, l2, parts = oracle.split_kv_decode(q, k, v, c["seqlens"], c["W"], dtype="f64")
        if not (_close(o1, out_ref) and _close(l1, lse_ref) and _close(o2, out_ref)
                and _close(l2, lse_ref)):
            return False
        if "combined_partial" in c:
            cp = c["combined_partial"]
            O, m, l = oracle.online_softmax_combine(parts[(0, 0)], c["d"])
            if not (_close(O, _arr(cp["O"])) and _close(m, _ev(cp["m"])) and _close(l, _ev(cp["l"]))):
                return False
    return True


def brute_force(q, k, v, seqlens, scale):
    """Pure-Python attention: lse = ln(fsum exp(s_j)) with no max shift; out = fsum softmax_j v_j."""
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    start = 0
    for b in range(B):
        L = int(seqlens[b])
        for h in range(Hq):
            g = h // G
            s = [scale * math.fsum(float(q[b, h, t]) * float(k[start + j, g, t]) for t in range(d))
                 for j in range(L)]
            if L == 0:
                lse[b, h] = -math.inf
                continue
            z = math.log(math.fsum(math.exp(x) for x in s))
            lse[b, h] = z
            for t in range(d):
                out[b, h, t] = math.fsum(math.exp(s[j] - z) * float(v[start + j, g, t]) for j in range(L))
        start += L
    return out, lse


def check_brute_force(seed=0, n_cases=12):
    rs = np.random.default_rng(seed)
    for _ in range(n_cases):
        Hkv = int(rs.integers(1, 3))
        G = int(rs.choice([1, 2, 4]))
        B = int(rs.integers(1, 3))
        d = int(rs.integers(1, 5))
        seqlens = rs.integers(0, 9, size=B)
        N = int(seqlens.sum())
        q = _rand_f64(rs, (B, Hq := Hkv * G, d), 1.5)
        k = _rand_f64(rs, (N, Hkv, d), 1.5)
        v = _rand_f64(rs, (N, Hkv, d))
        scale = 1.0 / math.sqrt(d)
        ob, lb = brute_force(q, k, v, seqlens, scale)
        o1, l1 = oracle.decode_reference(q, k, v, seqlens, dtype="f64")
        W = int(rs.integers(1, 10))
        o2, l2, _ = oracle.split_kv_decode(q, k, v, seqlens, W, dtype="f64")
        if not (_close(o1, ob, 1e-12) and _close(l1, lb, 1e-12) and _close(o2, ob, 1e-12)
                and _close(l2, lb, 1e-12)):
            return False
    return True


def _medium_problem(seed, B=2, Hq=4, Hkv=2, d=16, lens=(37, 91), dtype="f16"):
    return workloads.make_problem("medium", B, Hq, Hkv, d, list(lens), 1, dtype, seed)


def check_split_matches_definition(seed=1, Ws=(1, 2, 3, 7, 37, 200)):
    for dtype in ("f16", "bf16"):
        p = _medium_problem(seed, dtype=dtype)
        o_ref, l_ref = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, dtype)
        for W in Ws:
            o, l, _ = oracle.split_kv_decode(p.q, p.k, p.v, p.seqlens, W, dtype)
            if not (_close(o, o_ref, 1e-12) and _close(l, l_ref, 1e-12)):
                return False
    return True


def check_permutation_invariance(seed=2):
    p = _medium_problem(seed, lens=(64, 50))
    rs = np.random.default_rng(seed)
    o0, l0, _ = oracle.split_kv_decode(p.q, p.k, p.v, p.seqlens, 8, p.dtype)
    for _ in range(5):
        o1, l1, _ = oracle.split_kv_decode(p.q, p.k, p.v, p.seqlens, 8, p.dtype,
                                           order=lambda b, h, n: rs.permutation(n))
        if not (_close(o0, o1, 1e-12) and _close(l0, l1, 1e-12)):
            return False
    return True


def check_closed_forms(seed=3):
    rs = np.random.default_rng(seed)
    d, Hkv, G = 8, 2, 2
    Hq = Hkv * G
    scale = 1.0 / math.sqrt(d)
    # L = 1: out = V_0, lse = the single logit.
    q = rs.standard_normal((1, Hq, d))
    k = rs.standard_normal((1, Hkv, d))
    v = rs.standard_normal((1, Hkv, d))
    for W in (1, 3):
        o, l, _ = oracle.split_kv_decode(q, k, v, [1], W, dtype="f64")
        o2, l2 = oracle.decode_reference(q, k, v, [1], dtype="f64")
        for h in range(Hq):
            s0 = scale * float(np.dot(q[0, h], k[0, h // G]))
            if not (_close(o[0, h], v[0, h // G]) and _close(o2[0, h], v[0, h // G])
                    and abs(l[0, h] - s0) <= TOL and abs(l2[0, h] - s0) <= TOL):
                return False
    # All V rows equal to r: out = r.
    L = 57
    q = rs.standard_normal((1, Hq, d))
    k = rs.standard_normal((L, Hkv, d)) * 3
    r = rs.standard_normal((Hkv, d))
    v = np.broadcast_to(r, (L, Hkv, d)).copy()
    o, _ = oracle.decode_reference(q, k, v, [L], dtype="f64")
    o2, _, _ = oracle.split_kv_decode(q, k, v, [L], 5, dtype="f64")
    for h in range(Hq):
        if not (_close(o[0, h], r[h // G]) and _close(o2[0, h], r[h // G])):
            return False
    # q = 0: out = mean_j V_j and lse = ln L.
    q = np.zeros((1, Hq, d))
    v = rs.standard_normal((L, Hkv, d))
    o, l = oracle.decode_reference(q, k, v, [L], dtype="f64")
    o2, l2, _ = oracle.split_kv_decode(q, k, v, [L], 4, dtype="f64")
    for h in range(Hq):
        mean = v[:, h // G, :].mean(axis=0)
        if not (_close(o[0, h], mean) and _close(o2[0, h], mean)
                and abs(l[0, h] - math.log(L)) <= TOL and abs(l2[0, h] - math.log(L)) <= TOL):
            return False
    return True


def check_key_shift(seed=4):
    """K -> K + 1 c^T leaves out unchanged and adds scale * <q, c> to lse."""
    rs = np.random.default_rng(seed)
    B, Hkv, G, d = 2, 2, 2, 8
    Hq = Hkv * G
    lens = [23, 40]
    q = rs.standard_normal((B, Hq, d))
    k = rs.standard_normal((sum(lens), Hkv, d))
    v = rs.standard_normal((sum(lens), Hkv, d))
    c = rs.standard_normal((Hkv, d)) * 2.0
    o0, l0 = oracle.decode_reference(q, k, v, lens, dtype="f64")
    o1, l1 = oracle.decode_reference(q, k + c[None], v, lens, dtype="f64")
    o2, l2, _ = oracle.split_kv_decode(q, k + c[None], v, lens, 3, dtype="f64")
    scale = 1.0 / math.sqrt(d)
    for b in range(B):
        for h in range(Hq):
            shift = scale * float(np.dot(q[b, h], c[h // G]))
            if abs(l1[b, h] - (l0[b, h] + shift)) > 1e-11 or abs(l2[b, h] - (l0[b, h] + shift)) > 1e-11:
                return False
    return _close(o0, o1, 1e-11) and _close(o0, o2, 1e-11)


def check_convex_hull(seed=5):
    p = _medium_problem(seed, lens=(80, 33))
    o, _ = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    V = oracle.widen(p.v, p.dtype)
    G = p.Hq // p.Hkv
    start = 0
    for b in range(p.B):
        L = int(p.seqlens[b])
        for h in range(p.Hq):
            blk = V[start:start + L, h // G, :]
            if np.any(o[b, h] < blk.min(axis=0) - 1e-12) or np.any(o[b, h] > blk.max(axis=0) + 1e-12):
                return False
        start += L
    return True


def check_segment_rule():
    # The 4K case is four segments of 1024 tokens.
    if oracle.segment_bounds(4096, 4) != [(0, 1024), (1024, 2048), (2048, 3072), (3072, 4096)]:
        return False
    # W = ceil(L / 4096) gives segments of at most 4096 tokens.
    for L in (1024, 4095, 4096, 4097, 65536, 50001):
        W = -(-L // 4096)
        if max(e - s for s, e in oracle.segment_bounds(L, W)) > 4096:
            return False
    rs = np.random.default_rng(6)
    for _ in range(200):
        L = int(rs.integers(0, 300))
        W = int(rs.integers(1, 40))
        bnd = oracle.segment_bounds(L, W)
        if len(bnd) != W:
            return False
        S = -(-L // W) if L else 0
        pos = 0
        for s, e in bnd:
            if s != pos or e < s or e - s > S:
                return False
            pos = e
        if pos != L:
            return False
        lens = [e - s for s, e in bnd]
        if any(lens[i] < lens[i + 1] for i in range(W - 1)):
            return False
    return oracle.segment_bounds(0, 3) == [(0, 0)] * 3 and oracle.segment_bounds(3, 8)[3:] == [(3, 3)] * 5


def check_combine_algebra(seed=7):
    rs = np.random.default_rng(seed)
    d = 5
    ident = (np.zeros(d), -math.inf, 0.0)

    def rp():
        return rs.standard_normal(d), float(rs.standard_normal() * 4), float(rs.random() + 0.1)

    for _ in range(50):
        a, b, c = rp(), rp(), rp()
        ab = oracle.combine2(a, b)
        ba = oracle.combine2(b, a)
        l_ = oracle.combine2(oracle.combine2(a, b), c)
        r_ = oracle.combine2(a, oracle.combine2(b, c))
        for x, y in ((ab, ba), (l_, r_)):
            if not (_close(x[0], y[0], 1e-12) and abs(x[1] - y[1]) <= 1e-12 and abs(x[2] - y[2]) <= 1e-12):
                return False
        ai = oracle.combine2(a, ident)
        ia = oracle.combine2(ident, a)
        if not (_close(ai[0], a[0]) and ai[1] == a[1] and ai[2] == a[2]
                and _close(ia[0], a[0]) and ia[1] == a[1] and ia[2] == a[2]):
            return False
    # Combining two partials of one sequence equals the partial of the whole sequence.
    q = rs.standard_normal(d)
    K = rs.standard_normal((20, d))
    V = rs.standard_normal((20, d))
    whole = oracle.segment_partial(q, K, V, 0.5)
    halves = oracle.combine2(oracle.segment_partial(q, K[:7], V[:7], 0.5),
                             oracle.segment_partial(q, K[7:], V[7:], 0.5))
    return (_close(whole[0], halves[0], 1e-12) and abs(whole[1] - halves[1]) <= 1e-12
            and abs(whole[2] - halves[2]) <= 1e-12)


def check_bf16_bit_patterns():
    """bf16 inputs given as bit patterns of known values: 0x3F80=1, 0x4000=2, 0xC040=-3, 0x3E80=0.25."""
    vals = {0x3F80: 1.0, 0x4000: 2.0, 0xC040: -3.0, 0x3E80: 0.25}
    bits = np.array(list(vals), dtype=np.uint16)
    L, d = 4, 4
    q = np.zeros((1, 1, d), dtype=np.uint16)                       # +0.0
    k = np.zeros((L, 1, d), dtype=np.uint16)
    v = np.stack([np.roll(bits, j) for j in range(L)])[:, None, :]  # each column holds every value once
    o, l = oracle.decode_reference(q, k, v, [L], dtype="bf16")
    o2, l2, _ = oracle.split_kv_decode(q, k, v, [L], 2, dtype="bf16")
    mean = sum(vals.values()) / L
    return (_close(o, np.full((1, 1, d), mean)) and _close(o2, np.full((1, 1, d), mean))
            and abs(l[0, 0] - math.log(L)) <= TOL and abs(l2[0, 0] - math.log(L)) <= TOL)


def check_f16_bit_patterns():
    """fp16 inputs given as bit patterns of known values (IEEE binary16): 0x3C00 = 1,
    0xC000 = -2, 0x0001 = 2^-24 (smallest subnormal), 0x7BFF = 65504 (largest finite)."""
    vals = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -24, 0x7BFF: 65504.0}
    bits = np.array(list(vals), dtype=np.uint16)
    if not np.array_equal(oracle.widen(bits.view(np.float16), "f16"), np.array(list(vals.values()))):
        return False
    L, d = 4, 4
    q = np.zeros((1, 1, d), dtype=np.float16)
    k = np.zeros((L, 1, d), dtype=np.float16)
    v = np.stack([np.roll(bits, j) for j in range(L)])[:, None, :].view(np.float16)
    o, l = oracle.decode_reference(q, k, v, [L], dtype="f16")
    o2, l2, _ = oracle.split_kv_decode(q, k, v, [L], 3, dtype="f16")
    mean = (1.0 - 2.0 + 2.0 ** -24 + 65504.0) / L                  # exact in float64
    return (np.array_equal(o, np.full((1, 1, d), mean)) and _close(o2, np.full((1, 1, d), mean))
            and abs(l[0, 0] - math.log(L)) <= TOL and abs(l2[0, 0] - math.log(L)) <= TOL)


PINS = {
    "golden": check_golden,
    "bf16_bit_patterns": check_bf16_bit_patterns,
    "f16_bit_patterns": check_f16_bit_patterns,
    "brute_force": check_brute_force,
    "split_matches_definition": check_split_matches_definition,
    "permutation_invariance": check_permutation_invariance,
    "closed_forms": check_closed_forms,
    "key_shift": check_key_shift,
    "convex_hull": check_convex_hull,
    "segment_rule": check_segment_rule,
    "combine_algebra": check_combine_algebra,
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    assert PINS[name](), name


def test_library_sdpa_and_logsumexp():
    """Cross-check against torch's CPU scaled_dot_product_attention and logsumexp in float64."""
    torch = pytest.importorskip("torch")
    rs = np.random.default_rng(8)
    for (B, Hq, Hkv, d, L) in ((2, 8, 2, 16, 45), (1, 4, 4, 8, 130), (3, 6, 1, 32, 9)):
        q = rs.standard_normal((B, Hq, d))
        k = rs.standard_normal((B * L, Hkv, d)) * 2
        v = rs.standard_normal((B * L, Hkv, d))
        o, l = oracle.decode_reference(q, k, v, [L] * B, dtype="f64")
        G = Hq // Hkv
        tq = torch.from_numpy(q).unsqueeze(2)                                     # [B,Hq,1,d]
        tk = torch.from_numpy(k).reshape(B, L, Hkv, d).permute(0, 2, 1, 3)       # [B,Hkv,L,d]
        tv = torch.from_numpy(v).reshape(B, L, Hkv, d).permute(0, 2, 1, 3)
        tk = tk.repeat_interleave(G, dim=1)
        tv = tv.repeat_interleave(G, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[:, :, 0, :].numpy()
        assert np.max(np.abs(o - ref)) < 1e-12
        logits = torch.matmul(tq, tk.transpose(-1, -2))[:, :, 0, :] / math.sqrt(d)
        assert np.max(np.abs(l - torch.logsumexp(logits, dim=-1).numpy())) < 1e-12


def test_scipy_softmax_special_case():
    """With one KV head and Hq = 1 the weights are scipy's softmax of the logits."""
    special = pytest.importorskip("scipy.special")
    rs = np.random.default_rng(9)
    d, L = 16, 77
    q = rs.standard_normal((1, 1, d))
    k = rs.standard_normal((L, 1, d))
    V = np.eye(L)[:, None, :]                     # v_j = e_j, so out = the weight vector
    o, l = oracle.decode_reference(q, k, V, [L], dtype="f64")
    logits = (k[:, 0, :] @ q[0, 0]) / math.sqrt(d)
    assert np.max(np.abs(o[0, 0] - special.softmax(logits))) < 1e-14
    assert abs(l[0, 0] - special.logsumexp(logits)) < 1e-12


def test_sampled_heads_match_full():
    p = _medium_problem(10, lens=(31, 64))
    o, l = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype)
    picks = [(0, 1), (1, 3)]
    o2, l2 = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, p.dtype, heads=picks)
    o3, l3, _ = oracle.split_kv_decode(p.q, p.k, p.v, p.seqlens, 4, p.dtype, heads=picks)
    for b, h in picks:
        assert _close(o[b, h], o2[b, h]) and l[b, h] == l2[b, h]
        assert _close(o[b, h], o3[b, h], 1e-12) and abs(l[b, h] - l3[b, h]) < 1e-12
    assert np.isnan(o2[0, 0]).all()


def test_widen_is_exact():
    x = np.array([0.1, -3.5, 65504.0, 6e-8, 1e-3], dtype=np.float32)
    h = x.astype(np.float16)
    assert np.array_equal(oracle.widen(h, "f16"), h.astype(np.float64))
    bits = workloads.f32_to_bf16_bits(x)
    w = oracle.widen(bits, "bf16")
    # bf16 keeps the top 16 bits of the rounded float32
    assert np.array_equal(w.astype(np.float32).view(np.uint32) & 0xFFFF, np.zeros(5, np.uint32))
    assert np.all(np.abs(w - x) <= np.abs(x) * 2.0 ** -8)


# ---------------------------------------------------------------------------
# Planted mistakes: each must make at least one pin fail.
# ---------------------------------------------------------------------------

def _bad_combine_no_rescale(a, b):
    Oa, ma, la = a
    Ob, mb, lb = b
    if ma == -math.inf:
        return Ob, mb, lb
    if mb == -math.inf:
        return Oa, ma, la
    M = max(ma, mb)
    ea, eb = math.exp(ma - M), math.exp(mb - M)
    return Oa + Ob * eb, M, la * ea + lb * eb          # dropped e^{m_a - M} on O_a


def _bad_combine_sign(a, b):
    Oa, ma, la = a
    Ob, mb, lb = b
    if ma == -math.inf:
        return Ob, mb, lb
    if mb == -math.inf:
        return Oa, ma, la
    M = max(ma, mb)
    ea, eb = math.exp(M - ma), math.exp(mb - M)        # wrong sign in one exponent
    return Oa * ea + Ob * eb, M, la * ea + lb * eb


def _bad_segments_drop_last(L, W):
    b = fd_oracle.__dict__["_orig_segment_bounds"](L, W)
    return [(s, max(s, e - 1)) if i == W - 1 else (s, e) for i, (s, e) in enumerate(b)]


def _bad_segments_floor(L, W):
    S = L // W
    return [(min(w * S, L), min((w + 1) * S, L)) for w in range(W)]


def _bad_scale(d):
    return 1.0 / d


def _bad_partial_normalised(q_h, K_seg, V_seg, scale):
    O, m, l = fd_oracle.__dict__["_orig_segment_partial"](q_h, K_seg, V_seg, scale)
    return (O / l if l else O), m, l                    # normalised O combined as if unnormalised


def _bad_widen_bf16_low_half(x, dtype):
    if dtype == "bf16":
        return np.asarray(x, dtype=np.uint16).astype(np.float64)
    return fd_oracle.__dict__["_orig_widen"](x, dtype)


def _bad_finalize_log2(O, m, l):
    if l == 0.0:
        return np.zeros_like(O), -math.inf
    return O / l, m + math.log2(l)


MUTATIONS = {
    "combine_drops_rescale": ("combine2", _bad_combine_no_rescale),
    "combine_wrong_sign": ("combine2", _bad_combine_sign),
    "segments_drop_last_token": ("segment_bounds", _bad_segments_drop_last),
    "segments_floor_length": ("segment_bounds", _bad_segments_floor),
    "scale_one_over_d": ("default_scale", _bad_scale),
    "partial_normalised": ("segment_partial", _bad_partial_normalised),
    "bf16_widen_wrong": ("widen", _bad_widen_bf16_low_half),
    "lse_log2": ("finalize", _bad_finalize_log2),
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, monkeypatch):
    attr, bad = MUTATIONS[mutation]
    monkeypatch.setitem(fd_oracle.__dict__, "_orig_" + attr, getattr(fd_oracle, attr))
    monkeypatch.setattr(fd_oracle, attr, bad)
    monkeypatch.setattr(oracle, attr, bad, raising=False)
    failed = []
    for name, check in PINS.items():
        try:
            ok = check()
        except Exception:
            ok = False
        if not ok:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mutation}"


def test_paged_gather_round_trip():
    """A block table means: token t of sequence b is row t % P of page table[b][t // P]."""
    for page_size in (16, 64, 256):
        p = workloads.make_problem("paged", 4, 8, 2, 16, [0, 1, 300, 1025], [1, 2, 3, 4], "f16",
                                   seed=page_size)
        kp, vp, table = workloads.to_paged(p, page_size)
        k, v = oracle.gather_paged(kp, vp, table, p.seqlens, page_size)
        assert np.array_equal(k, p.k) and np.array_equal(v, p.v)
        # every used page appears once; spare pages are not referenced
        used = table[table >= 0]
        assert len(set(used.tolist())) == len(used) and len(used) == kp.shape[0] - 3


def test_e4m3_widening_known_codes():
    """OCP FP8 E4M3 codes of known values, and the round trip through the generator."""
    codes = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0x01: 2.0 ** -9,
             0x08: 2.0 ** -6, 0x07: 7 * 2.0 ** -9, 0xB8: -1.0, 0xC4: -3.0, 0x30: 0.5}
    arr = np.array(list(codes), dtype=np.uint8)
    assert np.array_equal(oracle.widen(arr, "e4m3"), np.array(list(codes.values())))
    assert np.isnan(oracle.widen(np.array([0x7F, 0xFF], dtype=np.uint8), "e4m3")).all()
    # every finite code survives the generator's rounding unchanged
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    vals = oracle.widen(finite, "e4m3").astype(np.float32)
    assert np.array_equal(workloads.f32_to_e4m3_bits(vals), finite)
    # rounding: halfway between 1.0 (0x38) and 1.125 (0x39) goes to the even code 0x38
    assert workloads.f32_to_e4m3_bits(np.array([1.0625], np.float32))[0] == 0x38
    assert workloads.f32_to_e4m3_bits(np.array([1.1875], np.float32))[0] == 0x3A
    assert workloads.f32_to_e4m3_bits(np.array([1000.0], np.float32))[0] == 0x7E


def test_e4m3_kv_split_matches_definition():
    p = workloads.with_e4m3_kv(workloads.make_problem("fp8", 2, 8, 2, 16, [77, 40], 3, "f16", seed=3))
    o1, l1 = oracle.decode_reference(p.q, p.k, p.v, p.seqlens, "f16", kv_dtype="e4m3")
    o2, l2, _ = oracle.split_kv_decode(p.q, p.k, p.v, p.seqlens, 5, "f16", kv_dtype="e4m3")
    assert _close(o1, o2, 1e-12) and _close(l1, l2, 1e-12)
    # the brute force on the widened values agrees
    ob, lb = brute_force(oracle.widen(p.q, "f16"), oracle.widen(p.k, "e4m3"),
                         oracle.widen(p.v, "e4m3"), p.seqlens, 1 / math.sqrt(16))
    assert _close(o1, ob, 1e-12) and _close(l1, lb, 1e-12)
