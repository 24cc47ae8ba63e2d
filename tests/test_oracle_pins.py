"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle (``oracle/``) against what the mathematics or the
pages fix: an exact brute force in 50-digit decimal arithmetic, closed forms,
invariants, a separately written streaming (m, d, o) implementation, torch's
CPU float64 SDPA, and the layout constants printed in the pages' listings.
``test_oracle_mutants`` then plants plausible mistakes in copies of the C
source and checks that these pins catch every one.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")


def rnd16(shape, seed, sigma=1.0):
    return synth.normal_fp16(shape, sigma, seed, 7)


def brute_decimal(q, k, v, scale, causal, prec=50):
    """Direct softmax without max shift, every step in 50-digit decimals.

    fp16 inputs and the double scale convert to Decimal exactly; products and
    sums of the tiny cases stay exact at this precision, so the only rounding
    is in exp, ln and the division, at ~1e-50.
    """
    getcontext().prec = prec
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    qd = q.astype(np.float64)
    kd = k.astype(np.float64)
    vd = v.astype(np.float64)
    sc = Decimal(float(scale))
    O = np.zeros((B, H, Nq, D))
    L = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                keys = range(min(i + 1, Nk)) if causal else range(Nk)
                e = {}
                for j in keys:
                    dot = sum(Decimal(float(qd[b, h, i, d])) * Decimal(float(kd[b, h, j, d]))
                              for d in range(D))
                    e[j] = (sc * dot).exp()
                Z = sum(e.values())
                for c in range(D):
                    O[b, h, i, c] = float(sum(e[j] * Decimal(float(vd[b, h, j, c])) for j in keys) / Z)
                L[b, h, i] = float(Z.ln())
    return O, L


TINY = [
    # B, H, Nq, Nk, D, causal, sigma
    (1, 1, 1, 1, 1, False, 1.0),
    (1, 1, 3, 5, 4, False, 1.0),
    (2, 2, 5, 3, 8, False, 1.5),
    (1, 2, 7, 7, 8, True, 1.0),
    (2, 1, 9, 4, 3, True, 2.0),
    (1, 1, 4, 9, 5, True, 1.0),
]


@pytest.mark.parametrize("B,H,Nq,Nk,D,causal,sigma", TINY)
def test_brute_force_decimal(B, H, Nq, Nk, D, causal, sigma):
    seed = B * 1000 + Nq * 100 + Nk * 10 + D
    q = rnd16((B, H, Nq, D), seed, sigma)
    k = rnd16((B, H, Nk, D), seed + 1, sigma)
    v = rnd16((B, H, Nk, D), seed + 2)
    scale = 1.0 / math.sqrt(D)
    O, L = oracle.attn_full(q, k, v, scale, causal)
    Ob, Lb = brute_decimal(q, k, v, scale, causal)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-13)


def test_half_decode_exhaustive():
    """All 65536 binary16 patterns decode exactly as numpy's float16 -> float64."""
    lib = oracle.default()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("causal", [False, True])
def test_q_zero_gives_mean_of_v(causal):
    """Q = 0: every score is 0, so O_i is the mean of V over the admissible
    keys (a prefix mean when causal) and LSE_i = ln |J_i|."""
    B, H, Nq, Nk, D = 2, 3, 19, 17, 16
    q = np.zeros((B, H, Nq, D), np.float16)
    k = rnd16((B, H, Nk, D), 11)
    v = rnd16((B, H, Nk, D), 12)
    O, L = oracle.attn_full(q, k, v, 0.25, causal)
    vd = v.astype(np.float64)
    for i in range(Nq):
        n = min(i + 1, Nk) if causal else Nk
        np.testing.assert_allclose(O[:, :, i], vd[:, :, :n].mean(axis=2), rtol=0, atol=1e-14)
        np.testing.assert_allclose(L[:, :, i], math.log(n), rtol=0, atol=1e-14)


def test_scale_zero_is_uniform():
    B, H, Nq, Nk, D = 1, 2, 6, 11, 8
    q, k, v = (rnd16(s, 20 + t, 3.0) for t, s in
               enumerate([(B, H, Nq, D), (B, H, Nk, D), (B, H, Nk, D)]))
    O, L = oracle.attn_full(q, k, v, 0.0, False)
    np.testing.assert_allclose(O, np.broadcast_to(v.astype(np.float64).mean(axis=2, keepdims=True),
                                                  O.shape), rtol=0, atol=1e-14)
    np.testing.assert_allclose(L, math.log(Nk), rtol=0, atol=1e-14)


def test_single_key():
    """Nk = 1: softmax of one score is 1, so O = V_0 and LSE = s_0."""
    B, H, Nq, D = 2, 2, 5, 8
    q = rnd16((B, H, Nq, D), 31)
    k = rnd16((B, H, 1, D), 32)
    v = rnd16((B, H, 1, D), 33)
    scale = 0.3
    for causal in (False, True):
        O, L = oracle.attn_full(q, k, v, scale, causal)
        np.testing.assert_array_equal(O, np.broadcast_to(v.astype(np.float64), O.shape))
        s0 = scale * np.einsum("bhid,bhd->bhi", q.astype(np.float64), k[:, :, 0].astype(np.float64))
        np.testing.assert_allclose(L, s0, rtol=0, atol=1e-14)


def test_constant_v():
    B, H, Nq, Nk, D = 1, 2, 9, 13, 8
    q = rnd16((B, H, Nq, D), 41, 2.0)
    k = rnd16((B, H, Nk, D), 42, 2.0)
    v = np.full((B, H, Nk, D), -1.25, np.float16)
    O, _ = oracle.attn_full(q, k, v, 0.35, True)
    np.testing.assert_allclose(O, -1.25, rtol=0, atol=1e-14)


def test_key_shift_invariance():
    """Adding one vector c to every key row shifts row i's scores by the same
    constant scale*q_i.c: O is unchanged and LSE moves by exactly that much.
    Inputs are multiples of 1/8 so that K + c is exact in fp16."""
    g = np.random.default_rng(5)
    B, H, Nq, Nk, D = 1, 2, 7, 10, 8
    q = (g.integers(-16, 17, (B, H, Nq, D)) / 8).astype(np.float16)
    k = (g.integers(-24, 25, (B, H, Nk, D)) / 8).astype(np.float16)
    v = rnd16((B, H, Nk, D), 51)
    c = (g.integers(-16, 17, (D,)) / 8)
    k2 = (k.astype(np.float64) + c).astype(np.float16)
    assert np.array_equal(k2.astype(np.float64), k.astype(np.float64) + c)
    scale = 0.25
    for causal in (False, True):
        O1, L1 = oracle.attn_full(q, k, v, scale, causal)
        O2, L2 = oracle.attn_full(q, k2, v, scale, causal)
        shift = scale * np.einsum("bhid,d->bhi", q.astype(np.float64), c)
        np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L2, L1 + shift, rtol=0, atol=1e-12)


def test_probability_rows_sum_to_one():
    B, H, Nq, Nk, D = 1, 2, 33, 40, 16
    q = rnd16((B, H, Nq, D), 61, 3.0)
    k = rnd16((B, H, Nk, D), 62, 3.0)
    v = rnd16((B, H, Nk, D), 63)
    for causal in (False, True):
        _, _, P, _ = oracle.attn_rows(q, k, v, 0.25, causal, want_probs=True)
        assert np.all(P >= 0)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        if causal:
            i = np.arange(B * H * Nq) % Nq
            j = np.arange(Nk)
            assert np.all(P[j[None, :] > i[:, None]] == 0)


def test_key_permutation_invariance():
    B, H, Nq, Nk, D = 2, 1, 12, 21, 16
    q = rnd16((B, H, Nq, D), 71)
    k = rnd16((B, H, Nk, D), 72)
    v = rnd16((B, H, Nk, D), 73)
    perm = np.random.default_rng(7).permutation(Nk)
    O1, L1 = oracle.attn_full(q, k, v, 0.25, False)
    O2, L2 = oracle.attn_full(q, np.ascontiguousarray(k[:, :, perm]),
                              np.ascontiguousarray(v[:, :, perm]), 0.25, False)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_streaming_carrier_any_tiling_any_order(causal):
    """The (m, d, o) carrier folded over key tiles of random sizes and merged
    in random orders equals the materialised definition."""
    B, H, Nq, Nk, D = 1, 2, 9, 23, 8
    q = rnd16((B, H, Nq, D), 81, 2.0)
    k = rnd16((B, H, Nk, D), 82, 2.0)
    v = rnd16((B, H, Nk, D), 83)
    O, L = oracle.attn_full(q, k, v, 0.4, causal)
    g = np.random.default_rng(8)
    for _ in range(4):
        cuts = np.sort(g.choice(np.arange(1, Nk), size=g.integers(1, 6), replace=False))
        bounds = [0, *cuts.tolist(), Nk]
        order = g.permutation(len(bounds) - 1).tolist()
        Os, Ls = oracle.attn_streaming(q, k, v, 0.4, causal, bounds, order)
        np.testing.assert_allclose(Os, O, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Ls, L, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Nq,Nk,causal", [(8, 8, False), (8, 8, True), (5, 9, True), (9, 5, True), (6, 11, False)])
def test_torch_cpu_float64_sdpa(Nq, Nk, causal):
    torch = pytest.importorskip("torch")
    B, H, D = 2, 3, 16
    q = rnd16((B, H, Nq, D), 91)
    k = rnd16((B, H, Nk, D), 92)
    v = rnd16((B, H, Nk, D), 93)
    scale = 1 / math.sqrt(D)
    O, L = oracle.attn_full(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
    To = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:  # torch's is_causal: key j masked when j > i (top-left)
        s = s.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).triu(1), float("-inf"))
    TL = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(O, To.numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, TL.numpy(), rtol=0, atol=1e-13)


def test_layout_matches_pages_listing_strides():
    """One Q element at the flat offset the pages' SDPA_L listing gives for
    (batch 0, head h, row i, channel d) moves exactly that output row."""
    facts = json.load(open(GOLDEN))
    B, H, N, D = facts["sdpa_l"]["shape"]
    st = facts["sdpa_l_strides"]
    assert (st["head"], st["batch"], st["row"]) == (N * D, H * N * D, D)
    k = rnd16((B, H, N, D), 101)
    v = rnd16((B, H, N, D), 102)
    q = np.zeros(B * H * N * D, np.float16)
    h, i, d = 2, 77, 5
    q[0 * st["batch"] + h * st["head"] + i * st["row"] + d] = 4.0
    O, _ = oracle.attn_full(q.reshape(B, H, N, D), k, v, facts["default_scale_d64"]["value"], False)
    mean_v = v.astype(np.float64).mean(axis=2)
    moved = np.abs(O - mean_v[:, :, None, :]).max(axis=3) > 1e-12
    assert moved.sum() == 1 and moved[0, h, i]


def test_flop_formula_matches_pages_throughput():
    """4*B*H*N*N*D at the pages' 206 us on SDPA_P is their ~167 TFLOP/s."""
    facts = json.load(open(GOLDEN))
    B, H, N, D = facts["sdpa_p"]["shape"]
    tflops = 4 * B * H * N * N * D / (facts["sdpa_p_latency"]["us"] * 1e-6) / 1e12
    assert abs(tflops - facts["sdpa_p_latency"]["tflops_about"]) < 0.5


def test_row_subset_and_thread_count():
    B, H, Nq, Nk, D = 2, 2, 50, 37, 16
    q = rnd16((B, H, Nq, D), 111)
    k = rnd16((B, H, Nk, D), 112)
    v = rnd16((B, H, Nk, D), 113)
    O, L = oracle.attn_full(q, k, v, 0.25, True, nthreads=1)
    O8, L8 = oracle.attn_full(q, k, v, 0.25, True, nthreads=8)
    assert np.array_equal(O, O8) and np.array_equal(L, L8)
    rows = np.array([199, 3, 77, 150, 0, 101])
    o, lse, _ = oracle.attn_rows(q, k, v, 0.25, True, rows)
    assert np.array_equal(o, O.reshape(-1, D)[rows])
    assert np.array_equal(lse, L.reshape(-1)[rows])


def test_large_scores_do_not_overflow():
    """Scores of magnitude ~1e3 (exp overflows without the max shift)."""
    B, H, Nq, Nk, D = 1, 1, 4, 6, 4
    q = np.full((B, H, Nq, D), 40.0, np.float16)
    k = rnd16((B, H, Nk, D), 121, 10.0)
    v = rnd16((B, H, Nk, D), 122)
    O, L = oracle.attn_full(q, k, v, 1.0, False)
    s = 40.0 * k.astype(np.float64).sum(axis=3)[0, 0]
    j = int(np.argmax(s))
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    np.testing.assert_allclose(L[0, 0], s.max() + np.log(np.exp(s - s.max()).sum()), rtol=1e-15)
    if np.sort(s)[-1] - np.sort(s)[-2] > 50:
        np.testing.assert_allclose(O[0, 0], np.broadcast_to(v[0, 0, j].astype(np.float64), (Nq, D)), atol=1e-15)
