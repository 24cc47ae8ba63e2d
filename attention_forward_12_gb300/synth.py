"""Seeded synthetic inputs for the attention forward.

This module is shared by the tests, the benchmark and the CPU oracle's
callers; it holds no attention arithmetic, only the workload recipes and a
counter-based random generator.

Recipe: every entry of Q, K and V is drawn i.i.d. from N(0, sigma^2) with
numpy's Philox4x32 counter-based generator, drawn in float32, scaled by sigma
and rounded to fp16 with round-to-nearest-even.  The flat tensor is cut into
chunks of 2^24 entries; chunk c of tensor t (0 = Q, 1 = K, 2 = V) comes from
the generator keyed (seed, t * 2^32 + c), so the values do not depend on how
many threads draw them.  The pages draw their inputs with
``torch.randn(..., dtype=torch.float16)`` and no seed ("Learning
FlashAttention the Hard Way -- Part 2", the SDPA_P / SDPA_L definitions);
this keeps that distribution and makes it reproducible.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 24  # elements drawn per generator call


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    D: int
    causal: bool
    sigma_qk: float
    sigma_v: float
    seed: int

    @property
    def scale(self) -> float:
        """Default softmax scale 1/sqrt(D), as F.scaled_dot_product_attention."""
        return 1.0 / math.sqrt(self.D)

    @property
    def shape_q(self):
        return (self.B, self.H, self.Nq, self.D)

    @property
    def shape_kv(self):
        return (self.B, self.H, self.Nk, self.D)


# The five workloads of the forward: the pages' listing shape (SDPA_L), the
# pages' benchmark shape (SDPA_P), and three long-sequence D=128 shapes, the
# last with Q and K drawn from N(0, 3^2) so that the softmax is sharply peaked
# and the running row maximum keeps growing along the key stream.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("sdpa_l_1x4x128x64", 1, 4, 128, 128, 64, False, 1.0, 1.0, 1),
        Workload("sdpa_p_1x8x4096x64", 1, 8, 4096, 4096, 64, False, 1.0, 1.0, 2),
        Workload("long_1x16x8192x128", 1, 16, 8192, 8192, 128, False, 1.0, 1.0, 3),
        Workload("causal_2x16x16384x128", 2, 16, 16384, 16384, 128, True, 1.0, 1.0, 4),
        Workload("peaked_4x32x16384x128", 4, 32, 16384, 16384, 128, False, 3.0, 1.0, 5),
    ]
}


def normal_fp16(shape, sigma: float, seed: int, stream: int) -> np.ndarray:
    """fp16 array of i.i.d. N(0, sigma^2) entries from Philox keyed (seed, stream)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)

    def fill(c: int) -> None:
        gen = np.random.Generator(np.random.Philox(key=[int(seed), (int(stream) << 32) + c]))
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        x = gen.standard_normal(hi - lo, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        out[lo:hi] = x  # float32 -> float16, round to nearest even

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def make_qkv(B: int, H: int, Nq: int, Nk: int, D: int, seed: int,
             sigma_qk: float = 1.0, sigma_v: float = 1.0):
    """(q, k, v) as contiguous fp16 numpy arrays, [B,H,Nq,D] and [B,H,Nk,D]."""
    q = normal_fp16((B, H, Nq, D), sigma_qk, seed, 0)
    k = normal_fp16((B, H, Nk, D), sigma_qk, seed, 1)
    v = normal_fp16((B, H, Nk, D), sigma_v, seed, 2)
    return q, k, v


def _e4m3_positive_values() -> np.ndarray:
    """Magnitudes of the OCP FP8 E4M3 codes 0..126 (ascending): codes below 8
    are subnormal, c/8 * 2^-6; the others (1 + (c mod 8)/8) * 2^(c div 8 - 7).
    Code 127 is NaN."""
    c = np.arange(127)
    return np.where(c < 8, c / 8.0 * 2.0 ** -6, (1.0 + (c & 7) / 8.0) * 2.0 ** ((c >> 3) - 7))


def to_e4m3(x) -> np.ndarray:
    """E4M3 codes (uint8) nearest to x: round to nearest, ties to the even
    code, magnitudes above 448 saturate to 448 (as a "satfinite" conversion).
    Input rounding only -- it serves the generators below."""
    x = np.asarray(x, dtype=np.float64)
    vals = _e4m3_positive_values()
    a = np.minimum(np.abs(x), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, 126)
    lo = hi - 1
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == 0, 0, code)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def make_qkv_e4m3(B: int, H: int, Nq: int, Nk: int, D: int, seed: int,
                  sigma_qk: float = 1.0, sigma_v: float = 1.0):
    """(q, k, v) as E4M3 codes (uint8 numpy arrays): the fp16 draws of
    make_qkv rounded to the nearest E4M3 value."""
    return tuple(to_e4m3(x.astype(np.float64)) for x in make_qkv(B, H, Nq, Nk, D, seed, sigma_qk, sigma_v))


def workload_qkv(w: Workload):
    return make_qkv(w.B, w.H, w.Nq, w.Nk, w.D, w.seed, w.sigma_qk, w.sigma_v)


def sample_rows(B: int, H: int, Nq: int, n_random: int, seed: int,
                causal: bool = False, tile: int = 128, head_rows: int = 512) -> np.ndarray:
    """Flat row ids ``(b*H+h)*Nq + i`` for a sampled parity check.

    The first and the last ``head_rows`` rows of the first and of the last
    head, ``n_random`` uniformly drawn rows, and in every head visited the
    edge rows 0, 1, tile-1, tile, tile+1, Nq-1 (plus, when causal, the first
    and last row of each query tile of the first head).  Sorted and unique.
    """
    rows = set()
    heads = B * H
    for hd in {0, heads - 1}:
        rows.update(range(hd * Nq, hd * Nq + min(Nq, head_rows)))
        rows.update(range(hd * Nq + max(0, Nq - head_rows), (hd + 1) * Nq))
    gen = np.random.Generator(np.random.Philox(key=[int(seed), 99]))
    r = gen.integers(0, heads * Nq, size=n_random)
    rows.update(int(x) for x in r)
    for hd in {int(x) // Nq for x in r} | {0, heads - 1}:
        for i in (0, 1, tile - 1, tile, tile + 1, Nq - 1):
            if 0 <= i < Nq:
                rows.add(hd * Nq + i)
    if causal:
        for t0 in range(0, Nq, tile):
            rows.add(t0)
            rows.add(min(Nq - 1, t0 + tile - 1))
    return np.array(sorted(rows), dtype=np.int64)
