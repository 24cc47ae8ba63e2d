"""Pins of the oracle's 8-bit path (no GPU): the E4M3 decode against the
format's definition and against torch's float8_e4m3fn, the input encoder
against torch's rounding, and the E4M3 attention against a brute-force
computation on independently decoded values."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth


# (code, value) from the OCP 8-bit floating point definition of E4M3:
# sign bit 7, exponent bits 6-3 with bias 7, mantissa bits 2-0, exponent 0
# subnormal, S.1111.111 NaN, no infinities.
HAND = [(0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
        (0x0F, 1.875 * 2.0 ** -6), (0x38, 1.0), (0x3C, 1.5), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0),
        (0xB8, -1.0), (0xFE, -448.0)]


def test_e4m3_decode_hand_values():
    codes = np.array([c for c, _ in HAND], dtype=np.uint8)
    got = oracle.e4m3_to_double(codes)
    for (c, want), g in zip(HAND, got):
        assert g == want and math.copysign(1.0, g) == math.copysign(1.0, want), hex(c)
    assert np.isnan(oracle.e4m3_to_double(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_matches_torch_on_every_code():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_to_double(codes), ref, equal_nan=True)


def test_input_encoder_matches_torch_rounding():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 20.0, 150.0)])
    x = x[np.abs(x) <= 448.0]  # torch maps values past the top rounding boundary to NaN
    # exact ties between neighbouring codes go to the even code
    vals = oracle.e4m3_to_double(np.arange(127, dtype=np.uint8))
    ties = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([x, ties, -ties, [0.0, -0.0, 448.0, 460.0]])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.to_e4m3(x), ref)
    # beyond the largest finite value the encoder saturates (torch gives NaN)
    assert list(synth.to_e4m3(np.array([500.0, -1e9]))) == [0x7E, 0xFE]


def _brute(q8, k8, v8, scale, causal, qd, kd, vd):
    torch = pytest.importorskip("torch")
    dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    q, k, v = dec(q8) * qd, dec(k8) * kd, dec(v8) * vd
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    O = np.zeros((B, H, Nq, D))
    L = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                n = min(Nk, i + 1) if causal else Nk
                s = scale * (k[b, h, :n] @ q[b, h, i])
                e = np.exp(s - s.max())
                O[b, h, i] = (e[:, None] * v[b, h, :n]).sum(0) / e.sum()
                L[b, h, i] = s.max() + math.log(e.sum())
    return O, L


@pytest.mark.parametrize("causal", [False, True])
def test_e4m3_attention_against_brute_force(causal):
    if not hasattr(pytest.importorskip("torch"), "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    q8, k8, v8 = synth.make_qkv_e4m3(2, 2, 7, 9, 16, seed=11, sigma_qk=1.5)
    qd, kd, vd = 0.5, 2.0, 0.25
    O, L = oracle.attn_full_e4m3(q8, k8, v8, 0.3, causal, qd, kd, vd)
    Ob, Lb = _brute(q8, k8, v8, 0.3, causal, qd, kd, vd)
    assert np.allclose(O, Ob, rtol=0, atol=1e-12) and np.allclose(L, Lb, rtol=0, atol=1e-12)


def test_e4m3_attention_closed_forms():
    v8 = synth.to_e4m3(synth.normal_fp16((1, 1, 6, 8), 1.0, 12, 2).astype(np.float64))
    q8 = np.zeros((1, 1, 6, 8), dtype=np.uint8)  # Q = 0: uniform weights
    k8 = synth.to_e4m3(synth.normal_fp16((1, 1, 6, 8), 1.0, 12, 1).astype(np.float64))
    O, L = oracle.attn_full_e4m3(q8, k8, v8, 0.5, True, v_descale=3.0)
    v = oracle.e4m3_to_double(v8)
    for i in range(6):
        assert np.allclose(O[0, 0, i], 3.0 * v[0, 0, : i + 1].mean(0), rtol=0, atol=1e-14)
        assert abs(L[0, 0, i] - math.log(i + 1)) < 1e-14
