"""Plant plausible mistakes in copies of the C oracle; the pins must catch each.

Every mutant is a one-line edit of ``oracle/attn_oracle.c`` compiled into a
temporary library (on the CPU; nothing here touches the CUDA path).  A mutant
counts as caught when at least one of the pins of ``test_oracle_pins`` --
brute force in decimal arithmetic, the exact half decode, the Q = 0 closed
form, the single-key closed form -- disagrees with it.
"""
import math
import os

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from test_oracle_pins import brute_decimal

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "attn_oracle.c")

MUTANTS = {
    "dropped_scale": ("s[j] *= w->scale;", "s[j] *= 1.0;"),
    "causal_off_by_one": ("if (w->causal && i + 1 < nval) nval = i + 1;",
                          "if (w->causal && i + 2 < nval) nval = i + 2;"),
    "k_in_place_of_v": ("const double *vj = w->vd + j * D;", "const double *vj = w->kt + j * D;"),
    "exp_sign_flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "lse_drops_max": ("w->lse_out[slot] = m + log(dsum);", "w->lse_out[slot] = log(dsum);"),
    "wrong_query_row": ("const uint16_t *qh = w->q + w->head_q_offset + i * D;",
                        "const uint16_t *qh = w->q + w->head_q_offset + ((i + 1) % w->Nq) * D;"),
    "half_bias_off": ("mag = ldexp((double)(1024 + f), e - 25);", "mag = ldexp((double)(1024 + f), e - 24);"),
    "half_subnormal_scale": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "normaliser_off": ("const double pj = s[j] / dsum;", "const double pj = s[j] / (dsum + 1.0);"),
    "k_read_transposed": ("kt[d * Nk + j] = oracle_half_to_double(kh[j * D + d]);",
                          "kt[d * Nk + j] = oracle_half_to_double(kh[d * Nk + j]);"),
    "v_from_wrong_head": ("const uint16_t *vh = v + head * Nk * D;",
                          "const uint16_t *vh = v + ((head + 1) % (B * H)) * Nk * D;"),
}


def pins_catch(lib: oracle.OracleLib) -> bool:
    # exact half decode on a spread of patterns (normals, subnormals, signs)
    bits = np.array([0x0001, 0x03FF, 0x0400, 0x3C00, 0x3555, 0x7BFF, 0xC000, 0x8001], np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    if any(lib.half_to_double(int(b)) != r for b, r in zip(bits, ref)):
        return True
    # brute force in decimal arithmetic
    for (B, H, Nq, Nk, D, causal) in [(1, 2, 5, 7, 4, False), (1, 2, 7, 5, 4, True)]:
        q = synth.normal_fp16((B, H, Nq, D), 1.0, 3, 0)
        k = synth.normal_fp16((B, H, Nk, D), 1.0, 3, 1)
        v = synth.normal_fp16((B, H, Nk, D), 1.0, 3, 2)
        scale = 1 / math.sqrt(D)
        O, L = lib.attn_full(q, k, v, scale, causal)
        Ob, Lb = brute_decimal(q, k, v, scale, causal)
        if not (np.allclose(O, Ob, rtol=0, atol=1e-13) and np.allclose(L, Lb, rtol=0, atol=1e-13)):
            return True
    # Q = 0 closed form (prefix mean when causal)
    q = np.zeros((1, 1, 6, 4), np.float16)
    v = synth.normal_fp16((1, 1, 6, 4), 1.0, 4, 2)
    O, L = lib.attn_full(q, synth.normal_fp16((1, 1, 6, 4), 1.0, 4, 1), v, 0.5, True)
    for i in range(6):
        if not np.allclose(O[0, 0, i], v[0, 0, : i + 1].astype(np.float64).mean(0), atol=1e-14):
            return True
        if abs(L[0, 0, i] - math.log(i + 1)) > 1e-14:
            return True
    # single key: O = V_0, LSE = s_0
    q = synth.normal_fp16((1, 1, 3, 4), 1.0, 5, 0)
    k = synth.normal_fp16((1, 1, 1, 4), 1.0, 5, 1)
    v = synth.normal_fp16((1, 1, 1, 4), 1.0, 5, 2)
    O, L = lib.attn_full(q, k, v, 0.5, False)
    s0 = 0.5 * q[0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64)
    if not (np.allclose(O[0, 0], v[0, 0, 0].astype(np.float64), atol=0) and np.allclose(L[0, 0], s0, atol=1e-14)):
        return True
    return False


def test_unmutated_oracle_passes_the_pins(tmp_path):
    lib = oracle.OracleLib(oracle.build(force=True, src=SRC, out=str(tmp_path / "ok.so")))
    assert not pins_catch(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_oracle_mutants(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / f"{name}.c"
    mut.write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.build(force=True, src=str(mut), out=str(tmp_path / f"{name}.so")))
    assert pins_catch(lib), f"mutant {name} survived the pins"
