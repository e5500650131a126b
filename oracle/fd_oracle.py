"""fp64 CPU oracle for split-KV Flash Decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this module.  The CUDA
path never calls it, and it shares no code with the CUDA path: it takes plain
numpy arrays (as drawn by ``workloads``) and returns plain numpy arrays.

Source: "Eliminating Multi-GPU Performance Taxes" (review page):
  * notation table: Q is the Flash Decode query, K_r / V_r the local KV-cache
    shard of rank r, O_r^partial the partial attention output of rank r;
  * core equations, "Flash Decode global reduction":
    O_final = OnlineSoftmaxCombine(O_0^partial, ..., O_{W-1}^partial), and the
    associativity of the online softmax lets partials be combined in any order;
  * correctness check #5: combine order does not change the result
    (Milakov & Gimelshein, 2018).

The method reaches plain softmax attention exactly (up to rounding order), so
``decode_reference`` is that definition written out.  ``split_kv_decode``
follows the split method step by step (segment rule, per-segment partial,
OnlineSoftmaxCombine fold, final normalisation) and is pinned against the
definition by the tests.

Readings where the pages are silent:
  * logit scale 1/sqrt(d); lse is the natural log of sum_j exp(s_j) over the
    *scaled* logits s_j;
  * GQA: query head h reads KV head h // G with G = Hq / Hkv;
  * partial = (O unnormalised, m = max logit, l = sum exp(s - m));
  * segment w of a length-L sequence split W ways is
    [w*S, min((w+1)*S, L)) with S = ceil(L / W); trailing segments may be
    empty and then contribute the combine identity (0, -inf, 0);
  * an empty sequence (L = 0) yields out = 0 and lse = -inf.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -math.inf


# ---------------------------------------------------------------------------
# Input widening (exact): stored 16-bit values -> float64.
# ---------------------------------------------------------------------------

def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored fp16 values or bf16 bit patterns to float64."""
    if dtype == "f16":
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    if dtype == "e4m3":
        # OCP FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
        # subnormal (m/8 * 2^-6); code S.1111.111 is NaN; there are no infinities.
        c = np.asarray(x, dtype=np.uint8).astype(np.int64)
        e, m = (c >> 3) & 0xF, c & 0x7
        mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
        mag = np.where((e == 15) & (m == 7), np.nan, mag)
        return np.where(c & 0x80, -mag, mag)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def gather_paged(k_pool, v_pool, block_table, seqlens, page_size):
    """Contiguous [N, Hkv, d] K and V from a paged cache.

    Token t of sequence b lives in pool page block_table[b][t // page_size], row
    t % page_size.  (Layout only: no arithmetic of the method.)
    """
    ks, vs = [], []
    for b, L in enumerate(np.asarray(seqlens, dtype=np.int64)):
        for t0 in range(0, int(L), page_size):
            page = int(block_table[b][t0 // page_size])
            n = min(page_size, int(L) - t0)
            ks.append(k_pool[page, :n])
            vs.append(v_pool[page, :n])
    if not ks:
        shape = (0,) + tuple(k_pool.shape[2:])
        return np.zeros(shape, k_pool.dtype), np.zeros(shape, v_pool.dtype)
    return np.concatenate(ks), np.concatenate(vs)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _cu(seqlens) -> np.ndarray:
    seqlens = np.asarray(seqlens, dtype=np.int64)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int64)
    np.cumsum(seqlens, out=cu[1:])
    return cu


# ---------------------------------------------------------------------------
# Definition: single-query softmax attention (Flash Decode computes exactly this).
# ---------------------------------------------------------------------------

def decode_reference(q, k, v, seqlens, dtype="f16", scale=None, heads=None, kv_dtype=None):
    """Plain single-token attention, fp64.

    For each sequence b and query head h (KV head g = h // G):
      s_j   = scale * <q[b,h], K[cu_b + j, g]>           j = 0 .. L_b - 1
      M     = max_j s_j,  Lam = sum_j exp(s_j - M)
      out   = sum_j exp(s_j - M) V[cu_b + j, g] / Lam
      lse   = M + ln(Lam)
    Empty sequences give out = 0 and lse = -inf.

    ``heads`` (optional) is a list of (b, h) pairs; only those rows are computed
    and the rest are left as NaN (used to sample very large cases).  ``kv_dtype``
    is the storage type of K and V when it differs from q's (e.g. "e4m3").
    Returns ``(out [B,Hq,dv] float64, lse [B,Hq] float64)``; dv = v.shape[2]
    (equal to d in every decode case; the oracle does not require it).
    """
    B, Hq, d = q.shape
    Hkv, dv = k.shape[1], v.shape[2]
    G = Hq // Hkv
    scale = default_scale(d) if scale is None else float(scale)
    cu = _cu(seqlens)
    out = np.full((B, Hq, dv), np.nan)
    lse = np.full((B, Hq), np.nan)
    want = None if heads is None else {(int(b), int(h)) for b, h in heads}
    for b in range(B):
        L = int(cu[b + 1] - cu[b])
        for g in range(Hkv):
            hs = [h for h in range(g * G, (g + 1) * G) if want is None or (b, h) in want]
            if not hs:
                continue
            if L == 0:
                for h in hs:
                    out[b, h] = 0.0
                    lse[b, h] = NEG_INF
                continue
            K = widen(k[cu[b]:cu[b + 1], g, :], kv_dtype or dtype)  # [L, d]
            V = widen(v[cu[b]:cu[b + 1], g, :], kv_dtype or dtype)  # [L, d]
            Q = widen(q[b, hs, :], dtype)                       # [n, d]
            S = scale * (Q @ K.T)                               # [n, L]
            M = S.max(axis=1, keepdims=True)
            E = np.exp(S - M)
            Lam = E.sum(axis=1, keepdims=True)
            out[b, hs] = (E @ V) / Lam
            lse[b, hs] = (M + np.log(Lam))[:, 0]
    return out, lse


# ---------------------------------------------------------------------------
# The split method, step by step.
# ---------------------------------------------------------------------------

def segment_bounds(L: int, W: int):
    """Split [0, L) into W contiguous segments of length S = ceil(L / W).

    Segment w is [min(w*S, L), min((w+1)*S, L)); the last non-empty one may be
    shorter and any after it are empty.  (The pages shard the KV cache W ways,
    one shard per rank; the case list states "W segments of 1024" for L=4096
    and W = ceil(L/4096), which this rule reproduces.)
    """
    if W < 1:
        raise ValueError("W must be >= 1")
    S = -(-L // W) if L > 0 else 0
    return [(min(w * S, L), min((w + 1) * S, L)) for w in range(W)]


def segment_partial(q_h, K_seg, V_seg, scale):
    """Partial attention of one query head over one KV segment (textbook two-pass).

    Returns (O, m, l): O = sum_j exp(s_j - m) V_j (unnormalised), m = max_j s_j,
    l = sum_j exp(s_j - m).  An empty segment returns the combine identity
    (0, -inf, 0).
    """
    if K_seg.shape[0] == 0:
        return np.zeros(V_seg.shape[1]), NEG_INF, 0.0
    s = scale * (K_seg @ q_h)
    m = float(s.max())
    e = np.exp(s - m)
    return e @ V_seg, m, float(e.sum())


def combine2(a, b):
    """OnlineSoftmaxCombine of two partials (associative and commutative).

    (O, m, l) (+) (O', m', l') = (O e^{m-M} + O' e^{m'-M}, M, l e^{m-M} + l' e^{m'-M}),
    M = max(m, m').  The identity (0, -inf, 0) is handled without forming
    exp(-inf - (-inf)).
    """
    Oa, ma, la = a
    Ob, mb, lb = b
    if ma == NEG_INF:
        return Ob, mb, lb
    if mb == NEG_INF:
        return Oa, ma, la
    M = max(ma, mb)
    ea, eb = math.exp(ma - M), math.exp(mb - M)
    return Oa * ea + Ob * eb, M, la * ea + lb * eb


def online_softmax_combine(partials, d):
    """Left fold of ``combine2`` over the partials, starting from the identity."""
    acc = (np.zeros(d), NEG_INF, 0.0)
    for p in partials:
        acc = combine2(acc, p)
    return acc


def finalize(O, m, l):
    """Normalise a combined partial: out = O / l, lse = m + ln l (l = 0 -> 0, -inf)."""
    if l == 0.0:
        return np.zeros_like(O), NEG_INF
    return O / l, m + math.log(l)


def split_kv_decode(q, k, v, seqlens, W, dtype="f16", scale=None, order=None, heads=None,
                    kv_dtype=None):
    """Split-KV Flash Decode, literally: segments -> partials -> combine -> normalise.

    ``W`` is an int or a per-sequence array.  ``order(b, h, n)`` (optional)
    returns the order in which the n partials of (b, h) are combined (tests use
    it to permute them).  Returns ``(out, lse, partials)`` where ``partials`` maps
    (b, h) to the list of (O, m, l) per segment in segment order.
    """
    B, Hq, d = q.shape
    Hkv, dv = k.shape[1], v.shape[2]
    G = Hq // Hkv
    scale = default_scale(d) if scale is None else float(scale)
    Ws = np.broadcast_to(np.asarray(W, dtype=np.int64), (B,))
    cu = _cu(seqlens)
    out = np.full((B, Hq, dv), np.nan)
    lse = np.full((B, Hq), np.nan)
    parts_all = {}
    want = None if heads is None else {(int(b), int(h)) for b, h in heads}
    for b in range(B):
        L = int(cu[b + 1] - cu[b])
        bounds = segment_bounds(L, int(Ws[b]))
        for h in range(Hq):
            if want is not None and (b, h) not in want:
                continue
            g = h // G
            qh = widen(q[b, h, :], dtype)
            parts = []
            for (s0, s1) in bounds:
                K = widen(k[cu[b] + s0:cu[b] + s1, g, :], kv_dtype or dtype)
                V = widen(v[cu[b] + s0:cu[b] + s1, g, :], kv_dtype or dtype)
                parts.append(segment_partial(qh, K, V, scale))
            seq = parts if order is None else [parts[i] for i in order(b, h, len(parts))]
            O, m, l = online_softmax_combine(seq, dv)
            out[b, h], lse[b, h] = finalize(O, m, l)
            parts_all[(b, h)] = parts
    return out, lse, parts_all
