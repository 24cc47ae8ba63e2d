"""fp64 CPU oracle for the attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is independent of the CUDA path:
it never imports ``attention_forward_12_gb300`` and shares no code with it.

Two implementations live here and pin each other:

* :func:`attn_rows` / :func:`attn_full` -- the plain definition (C, fp64,
  ``attn_oracle.c``): materialised score row, max pass, exp-sum pass,
  normalise-and-PV pass, per "Learning FlashAttention the Hard Way -- Part 2",
  section "Move 0 -- Scalar Streaming Kernel" (the two-kernel naive lowering).
* :func:`attn_streaming` -- the streaming reduction of the same page: the
  carrier triple (m, d, o) updated key tile by key tile (section "Move 0",
  the FA-1 listing: m' = max(m, s), alpha = e^(m - m'), p = e^(s - m'),
  d <- d*alpha + p, o <- o*alpha + p*v, normalise o/d at the end), with tiles
  of arbitrary sizes combined in an arbitrary order by the merge of two
  carriers.  The page calls the reduction associative (its opening paragraph
  and "Relationship to FA-3 and FA-4": split-KV is "the monoid's split-K")
  but never prints the merge; the plain reading used here is
      (m1,d1,o1) (+) (m2,d2,o2) = (m, d1 e^(m1-m) + d2 e^(m2-m),
                                    o1 e^(m1-m) + o2 e^(m2-m)),  m = max(m1,m2).
  It is numpy fp64 and small-case only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the C oracle ``src`` into the shared library ``out`` (gcc, -O3).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    the oracle gives the same bits on x86-64 and aarch64 hosts.
    """
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-pthread", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _bits(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are fp16 arrays (or their uint16 bit patterns)")
    return np.ascontiguousarray(a)


class OracleLib:
    """ctypes view of one compiled copy of ``attn_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64 = ctypes.c_int64
        p = ctypes.c_void_p
        lib.oracle_attn_rows.restype = ctypes.c_int
        lib.oracle_attn_rows.argtypes = [p, p, p, i64, i64, i64, i64, i64,
                                         ctypes.c_double, ctypes.c_int, p, i64,
                                         p, p, p, ctypes.c_int]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        self._lib = lib
        self.path = path

    def half_to_double(self, bits: int) -> float:
        """Exact binary16 -> double decode of the C oracle."""
        return self._lib.oracle_half_to_double(int(bits) & 0xFFFF)

    def attn_rows(self, q, k, v, scale: float, causal: bool, rows=None,
                  nthreads: int = 0, want_probs: bool = False):
        """O and LSE (fp64) for selected query rows.

        q: fp16 [B,H,Nq,D]; k, v: fp16 [B,H,Nk,D] (numpy float16 or uint16
        bits).  rows: flat row ids ``(b*H + h)*Nq + i`` or None for every row.
        Returns (O [n,D], LSE [n], threads used), or with ``want_probs``
        (O, LSE, P [n,Nk], threads used).
        """
        q, k, v = _bits(q), _bits(k), _bits(v)
        B, H, Nq, D = q.shape
        Bk, Hk, Nk, Dk = k.shape
        if (Bk, Hk, Dk) != (B, H, D) or v.shape != k.shape:
            raise ValueError("shape mismatch between q, k, v")
        if rows is None:
            n = B * H * Nq
            rows_arr = None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            n = rows_arr.size
        o = np.empty((n, D), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        probs = np.empty((n, Nk), dtype=np.float64) if want_probs else None
        used = self._lib.oracle_attn_rows(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Nq, Nk, D,
            float(scale), int(bool(causal)),
            None if rows_arr is None else rows_arr.ctypes.data, n,
            o.ctypes.data, lse.ctypes.data,
            None if probs is None else probs.ctypes.data, int(nthreads))
        if used < 0:
            raise ValueError(f"oracle_attn_rows rejected its arguments ({used})")
        if want_probs:
            return o, lse, probs, used
        return o, lse, used

    def attn_full(self, q, k, v, scale: float, causal: bool, nthreads: int = 0):
        """O [B,H,Nq,D] and LSE [B,H,Nq] (fp64) for every row."""
        B, H, Nq, D = q.shape
        o, lse, _ = self.attn_rows(q, k, v, scale, causal, None, nthreads)
        return o.reshape(B, H, Nq, D), lse.reshape(B, H, Nq)


def default() -> OracleLib:
    """The oracle built from ``attn_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def half_to_double(bits: int) -> float:
    return default().half_to_double(bits)


def attn_rows(q, k, v, scale: float, causal: bool, rows=None, nthreads: int = 0,
              want_probs: bool = False):
    return default().attn_rows(q, k, v, scale, causal, rows, nthreads, want_probs)


def attn_full(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """O [B,H,Nq,D] and LSE [B,H,Nq] (fp64) for every row."""
    return default().attn_full(q, k, v, scale, causal, nthreads)


# ---------------------------------------------------------------------------
# 8-bit inputs: OCP FP8 E4M3.
# ---------------------------------------------------------------------------

def e4m3_to_double(codes) -> np.ndarray:
    """Exact value of OCP FP8 E4M3 codes (the "fn" variant of the OCP 8-bit
    floating point specification: no infinities, S.1111.111 is NaN).  Bit 7
    is the sign, bits 6-3 the exponent E (bias 7), bits 2-0 the mantissa M:
    E = 0 gives (-1)^S * M/8 * 2^-6, otherwise (-1)^S * (1 + M/8) * 2^(E-7)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    return np.where((c & 0x7F) == 0x7F, np.nan, sign * mag)


def _e4m3_as_fp16(codes) -> np.ndarray:
    """E4M3 codes as fp16 arrays: every E4M3 value is an fp16 value (3 of the
    10 mantissa bits, exponents -9 .. 8), so the conversion is exact."""
    d = e4m3_to_double(codes)
    h = d.astype(np.float16)
    if not np.array_equal(h.astype(np.float64), d, equal_nan=True):
        raise AssertionError("E4M3 -> fp16 must be exact")
    return h


def attn_rows_e4m3(q8, k8, v8, scale: float, causal: bool, q_descale: float = 1.0,
                   k_descale: float = 1.0, v_descale: float = 1.0, rows=None, nthreads: int = 0,
                   want_probs: bool = False):
    """O and LSE (fp64) on E4M3 inputs: the plain definition over the exact
    values q_descale*Q, k_descale*K, v_descale*V, i.e. the fp16 oracle on the
    decoded codes with scale * q_descale * k_descale, and O times v_descale.
    Returns (O, LSE, threads) or, with want_probs, (O, LSE, P, threads), P
    the softmax weights [n, Nk]."""
    q, k, v = (_e4m3_as_fp16(x) for x in (q8, k8, v8))
    res = attn_rows(q, k, v, float(scale) * float(q_descale) * float(k_descale), causal, rows, nthreads,
                    want_probs)
    return (res[0] * float(v_descale),) + tuple(res[1:])


def attn_full_e4m3(q8, k8, v8, scale: float, causal: bool, q_descale: float = 1.0,
                   k_descale: float = 1.0, v_descale: float = 1.0, nthreads: int = 0):
    """O [B,H,Nq,D] and LSE [B,H,Nq] (fp64) for every row, E4M3 inputs."""
    B, H, Nq, D = np.asarray(q8).shape
    o, lse, _ = attn_rows_e4m3(q8, k8, v8, scale, causal, q_descale, k_descale, v_descale, None, nthreads)
    return o.reshape(B, H, Nq, D), lse.reshape(B, H, Nq)


# ---------------------------------------------------------------------------
# Streaming carrier (m, d, o) -- a second, separately written implementation.
# ---------------------------------------------------------------------------

def carrier_of_tile(s: np.ndarray, vt: np.ndarray):
    """Carrier of one key tile for one query row: fold keys one at a time.

    s: [n] scores of the tile's admissible keys, vt: [n, D] their V rows.
    Starts from the identity (m = -inf, d = 0, o = 0) and applies the page's
    per-key update m' = max(m, s_j), alpha = e^(m - m'), p = e^(s_j - m'),
    d <- d*alpha + p, o <- o*alpha + p*v_j.
    """
    m = -np.inf
    d = 0.0
    o = np.zeros(vt.shape[1], dtype=np.float64)
    for j in range(s.shape[0]):
        m_new = max(m, s[j])
        alpha = np.exp(m - m_new) if m != -np.inf else 0.0
        p = np.exp(s[j] - m_new)
        d = d * alpha + p
        o = o * alpha + p * vt[j]
        m = m_new
    return m, d, o


def carrier_merge(a, b):
    """(m1,d1,o1) (+) (m2,d2,o2): rescale both to the larger max and add."""
    m1, d1, o1 = a
    m2, d2, o2 = b
    if m1 == -np.inf:
        return b
    if m2 == -np.inf:
        return a
    m = max(m1, m2)
    e1 = np.exp(m1 - m)
    e2 = np.exp(m2 - m)
    return m, d1 * e1 + d2 * e2, o1 * e1 + o2 * e2


def attn_streaming(q, k, v, scale: float, causal: bool, tile_bounds, order):
    """O and LSE from carriers of key tiles merged in a given order.

    tile_bounds: increasing key indices [0, b1, ..., Nk] cutting the keys of
    every row into tiles; order: a permutation of the tile indices giving the
    order in which tile carriers are merged.  Small inputs only (pure Python
    over rows and keys).
    """
    qd = _bits(q).view(np.float16).astype(np.float64)
    kd = _bits(k).view(np.float16).astype(np.float64)
    vd = _bits(v).view(np.float16).astype(np.float64)
    B, H, Nq, D = qd.shape
    Nk = kd.shape[2]
    O = np.zeros((B, H, Nq, D))
    L = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                nval = min(i + 1, Nk) if causal else Nk
                acc = (-np.inf, 0.0, np.zeros(D))
                for t in order:
                    lo, hi = tile_bounds[t], min(tile_bounds[t + 1], nval)
                    if hi <= lo:
                        continue
                    s = np.array([scale * float(np.dot(qd[b, h, i], kd[b, h, j]))
                                  for j in range(lo, hi)])
                    acc = carrier_merge(acc, carrier_of_tile(s, vd[b, h, lo:hi]))
                m, d, o = acc
                O[b, h, i] = o / d
                L[b, h, i] = m + np.log(d)
    return O, L

