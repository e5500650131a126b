"""Seeded synthetic decode workloads.

One query token per sequence attends over a long KV cache that is split into
W segments ("Eliminating Multi-GPU Performance Taxes", review page, notation
table and the Flash Decode global-reduction equation).  The pages measure
Flash Decode on synthetic shapes only (batch 1, 96 query heads, head dim 128,
KV length 32K..2M, FP16; Flash Decode setup paragraph), so every workload here
is synthetic: q, K and V are standard-normal draws from a seeded generator,
stored in the 16-bit type of the case.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It only draws numbers and lays them out; it holds none of the
attention arithmetic (no scores, no softmax, no combine).

Layouts (all C-contiguous):
  q  [B, Hq, d]
  k  [N, Hkv, d]   sequence b occupies rows [cu[b], cu[b] + L_b), N = sum L_b
  v  [N, Hkv, d]
16-bit storage: ``np.float16`` for f16, ``np.uint16`` holding bf16 bit
patterns for bf16 (numpy has no bfloat16 type).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F16 = "f16"
BF16 = "bf16"

# Independent generator streams per tensor (q, K, V, spike positions, lengths).
_STREAM_Q, _STREAM_K, _STREAM_V, _STREAM_SPIKE, _STREAM_LEN = 1, 2, 3, 4, 5

_CHUNK = 1 << 25  # elements drawn per generator call (bounds fp32 temporaries)


@dataclass
class DecodeProblem:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    seqlens: np.ndarray          # int32 [B]
    W: np.ndarray                # int32 [B], segments per sequence
    dtype: str                   # "f16" | "bf16"
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    seed: int
    literal_w: bool = False      # run exactly W segments per sequence (no sub-chunks)
    notes: dict = field(default_factory=dict)
    kv_dtype: str = ""           # K/V storage type when it differs from q's ("e4m3")

    @property
    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.B + 1, dtype=np.int64)
        np.cumsum(self.seqlens.astype(np.int64), out=cu[1:])
        return cu

    @property
    def n_tokens(self) -> int:
        return int(self.seqlens.astype(np.int64).sum())

    @property
    def kv_type(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V that one decode must read."""
        return 2 * self.n_tokens * self.Hkv * self.d * (1 if self.kv_type == E4M3 else 2)

    def describe(self) -> dict:
        return {
            "workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv,
            "d": self.d, "dtype": self.dtype, "seed": self.seed,
            "L": (int(self.seqlens[0]) if self.B == 1 else
                  {"min": int(self.seqlens.min()), "max": int(self.seqlens.max()),
                   "sum": self.n_tokens}),
            "W": (int(self.W[0]) if np.all(self.W == self.W[0]) else
                  {"min": int(self.W.min()), "max": int(self.W.max()),
                   "sum": int(self.W.sum())}),
            "literal_w": self.literal_w, **({"kv_dtype": self.kv_dtype} if self.kv_dtype else {}),
            **self.notes,
        }


def rng(seed: int, stream: int) -> np.random.Generator:
    """Independent, reproducible stream ``stream`` of the workload seeded ``seed``."""
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


E4M3 = "e4m3"

# The 127 non-negative finite values of OCP FP8 E4M3 (codes 0x00 .. 0x7E), in code order.
_E4M3_POS = np.array(
    [m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
     for e in range(16) for m in range(8)][:127], dtype=np.float64)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to OCP FP8 E4M3 (nearest, ties to even code; saturate at 448); return the codes."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(_E4M3_POS, a, side="left").clip(0, 126)
    lo = (hi - 1).clip(0, 126)
    dlo, dhi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == F16:
        return x32.astype(np.float16)
    if dtype == BF16:
        return f32_to_bf16_bits(x32)
    if dtype == E4M3:
        return f32_to_e4m3_bits(x32)
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of the stored 16-bit values to float32."""
    if dtype == F16:
        return np.asarray(x, dtype=np.float16).astype(np.float32)
    if dtype == BF16:
        return bf16_bits_to_f32(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def normal(gen: np.random.Generator, shape, dtype: str, scale_rows=None) -> np.ndarray:
    """Standard-normal draw in float32, optionally scaling whole token rows, stored as ``dtype``.

    ``scale_rows`` is ``(row_indices, factor)``: those rows of the leading axis
    are multiplied by ``factor`` in float32 before the single rounding to 16 bits.
    """
    shape = tuple(int(s) for s in shape)
    total = int(np.prod(shape)) if shape else 1
    out = np.empty(total, dtype=np.float16 if dtype == F16 else np.uint16)
    row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    rows_hit = None
    if scale_rows is not None:
        rows_hit = (np.sort(np.asarray(scale_rows[0], dtype=np.int64)), np.float32(scale_rows[1]))
    chunk = max(row, (_CHUNK // row) * row)
    for start in range(0, total, chunk):
        stop = min(total, start + chunk)
        x = gen.standard_normal(stop - start, dtype=np.float32)
        if rows_hit is not None:
            r0, r1 = start // row, stop // row
            idx, factor = rows_hit
            sel = idx[(idx >= r0) & (idx < r1)]
            for r in sel:
                a = (int(r) - r0) * row
                x[a:a + row] *= factor
        out[start:stop] = to_storage(x, dtype)
    return out.reshape(shape)


def make_problem(name, B, Hq, Hkv, d, seqlens, W, dtype=F16, seed=0, literal_w=False,
                 k_spike_rows=None, k_spike_factor=20.0, notes=None) -> DecodeProblem:
    seqlens = np.asarray(seqlens, dtype=np.int32).reshape(B)
    W = np.broadcast_to(np.asarray(W, dtype=np.int32), (B,)).copy()
    N = int(seqlens.astype(np.int64).sum())
    q = normal(rng(seed, _STREAM_Q), (B, Hq, d), dtype)
    spike = None if k_spike_rows is None else (k_spike_rows, k_spike_factor)
    k = normal(rng(seed, _STREAM_K), (N, Hkv, d), dtype, scale_rows=spike)
    v = normal(rng(seed, _STREAM_V), (N, Hkv, d), dtype)
    return DecodeProblem(name, B, Hq, Hkv, d, seqlens, W, dtype, q, k, v, seed,
                         literal_w, dict(notes or {}))


_STREAM_PAGES = 6


def with_e4m3_kv(problem: DecodeProblem) -> DecodeProblem:
    """The same case with K and V rounded once to OCP FP8 E4M3 (q stays 16-bit).

    Per-tensor scales are 1: standard-normal values sit well inside E4M3's range
    (|x| <= 448).  A scaled cache folds its K scale into q and its V scale into out.
    """
    from dataclasses import replace
    k = f32_to_e4m3_bits(storage_to_f32(problem.k, problem.dtype))
    v = f32_to_e4m3_bits(storage_to_f32(problem.v, problem.dtype))
    return replace(problem, name=problem.name + "_kv_e4m3", k=k, v=v, kv_dtype=E4M3)


def to_paged(problem: DecodeProblem, page_size: int, spare_pages: int = 3, seed: int = None):
    """Scatter a problem's contiguous K/V into a shuffled page pool.

    Returns ``(k_pool, v_pool, block_table)``: pools ``[num_pages, page_size, Hkv, d]``
    and an int32 table ``[B, max_pages]`` (unused entries -1) whose row b lists the
    pool pages holding tokens ``[j*page_size, (j+1)*page_size)`` of sequence b.  Page
    order is a seeded permutation, with ``spare_pages`` pages that no sequence uses.
    Rows of a sequence's last page beyond its length are filled with random values.
    """
    seed = problem.seed if seed is None else seed
    gen = rng(seed, _STREAM_PAGES)
    lens = problem.seqlens.astype(np.int64)
    npg = (lens + page_size - 1) // page_size
    total = int(npg.sum()) + spare_pages
    max_pages = max(1, int(npg.max()) if len(npg) else 1)
    perm = gen.permutation(total)
    shape = (total, page_size, problem.Hkv, problem.d)
    k_pool = normal(gen, shape, problem.dtype)
    v_pool = normal(gen, shape, problem.dtype)
    if problem.kv_type == E4M3:
        k_pool = f32_to_e4m3_bits(storage_to_f32(k_pool, problem.dtype))
        v_pool = f32_to_e4m3_bits(storage_to_f32(v_pool, problem.dtype))
    table = np.full((problem.B, max_pages), -1, dtype=np.int32)
    cu = problem.cu_seqlens
    nxt = 0
    for b in range(problem.B):
        for j in range(int(npg[b])):
            page = int(perm[nxt])
            nxt += 1
            table[b, j] = page
            t0 = j * page_size
            t1 = min(int(lens[b]), t0 + page_size)
            k_pool[page, :t1 - t0] = problem.k[cu[b] + t0:cu[b] + t1]
            v_pool[page, :t1 - t0] = problem.v[cu[b] + t0:cu[b] + t1]
    return k_pool, v_pool, table


# ---------------------------------------------------------------------------
# The five decode cases (one fixed seed each, 1000 + index).
# ---------------------------------------------------------------------------

def mha8_d64_L4k_W4(seed: int = 1000) -> DecodeProblem:
    """B=1, Hq=Hkv=8, d=64, L=4096 split into W=4 segments of 1024; fp16 N(0,1)."""
    return make_problem("mha8_d64_L4k_W4", 1, 8, 8, 64, [4096], 4, F16, seed)


def gqa4_d128_L32k_W8(seed: int = 1001) -> DecodeProblem:
    """B=1 decode, Hq=32 / Hkv=8 (4 query heads per KV head), d=128, L=32768, W=8; fp16 N(0,1)."""
    return make_problem("gqa4_d128_L32k_W8", 1, 32, 8, 128, [32768], 8, F16, seed)


def gqa8_d128_L128k_W8_spiky(seed: int = 1002, dtype: str = F16) -> DecodeProblem:
    """B=1, Hq=64 / Hkv=8, d=128, L=131072, W=8; fp16 N(0,1) with 0.1% of key rows x20.

    round(0.001 * L) = 131 token positions are drawn without replacement from
    their own stream; every KV head of K at those positions is multiplied by 20
    in float32 before rounding once to fp16.  V is untouched.  ``dtype="bf16"``
    gives the same draw rounded to bf16 instead (not one of the five cases).
    """
    L = 131072
    n_spike = int(round(0.001 * L))
    rows = rng(seed, _STREAM_SPIKE).choice(L, size=n_spike, replace=False)
    name = "gqa8_d128_L128k_W8_spiky" + ("" if dtype == F16 else "_" + dtype)
    return make_problem(name, 1, 64, 8, 128, [L], 8, dtype, seed,
                        k_spike_rows=rows, k_spike_factor=20.0,
                        notes={"k_spike_rows": n_spike, "k_spike_factor": 20.0})


def ragged16_gqa4_d128(seed: int = 1003) -> DecodeProblem:
    """B=16 ragged batch, Hq=32 / Hkv=8, d=128, L_b uniform in [1024, 65536], W_b = ceil(L_b/4096)."""
    lens = rng(seed, _STREAM_LEN).integers(1024, 65536, size=16, endpoint=True).astype(np.int32)
    W = ((lens.astype(np.int64) + 4095) // 4096).astype(np.int32)
    return make_problem("ragged16_gqa4_d128", 16, 32, 8, 128, lens, W, F16, seed)


def batch64_gqa4_d128_L8k_bf16(W: int = 1, seed: int = 1004, B: int = 64) -> DecodeProblem:
    """B=64, Hq=32 / Hkv=8, d=128, L=8192 each, bf16 N(0,1); W in {1,2,4,8,16}, exactly W segments.

    The inputs do not depend on W (same seed), so a W sweep runs on identical data.
    ``B`` < 64 gives the first B sequences of the same draw (a smaller case of the
    same kernel, e.g. for a profiler capture); it is not one of the five cases.
    """
    name = f"batch{B}_gqa4_d128_L8k_bf16_W{W}"
    return make_problem(name, B, 32, 8, 128, [8192] * B, W, BF16, seed, literal_w=True)


def gqa16_d128_L32k_W8(seed: int = 1005) -> DecodeProblem:
    """B=1, Hq=128 / Hkv=8 (16 query heads per KV head), d=128, L=32768, W=8; fp16 N(0,1).

    Not one of the five decode cases: a larger GQA group for the tensor-core path.
    """
    return make_problem("gqa16_d128_L32k_W8", 1, 128, 8, 128, [32768], 8, F16, seed)


CASES = {
    "mha8_d64_L4k_W4": mha8_d64_L4k_W4,
    "gqa4_d128_L32k_W8": gqa4_d128_L32k_W8,
    "gqa8_d128_L128k_W8_spiky": gqa8_d128_L128k_W8_spiky,
    "ragged16_gqa4_d128": ragged16_gqa4_d128,
    "batch64_gqa4_d128_L8k_bf16": batch64_gqa4_d128_L8k_bf16,
}

# Extra shapes (not among the five decode cases).
EXTRA = {
    "gqa16_d128_L32k_W8": gqa16_d128_L32k_W8,
}

W_SWEEP = (1, 2, 4, 8, 16)
