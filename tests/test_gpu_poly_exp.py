"""The FMA-pipe 2^x ("the FMA-emulated exp" the page credits to
FlashAttention-4, "Relationship to FA-3 and FA-4") on the device: the
routine on its own against exact powers of two, and a forward that sends a
quarter of its exponentials to it against the fp64 oracle.  The forward
itself keeps every exponential on the exponential unit (on GB300 the split
measured slower), so these tests are what runs the device code."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from gpu_common import compare, torch_cuda

pytestmark = pytest.mark.gpu

# The routine's stated bound on [-126, 127]; its fp32 evaluation on the CPU
# reaches 3.7e-6 (tests/test_exp2_poly.py).
REL_BOUND = 4e-6


@pytest.fixture(scope="module")
def attn():
    torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    attn.load_library()
    return attn


def test_exp2_poly_on_the_device_is_within_its_bound(attn):
    import torch
    gen = np.random.Generator(np.random.Philox(key=[7, 0]))
    grid = np.linspace(-126.0, 127.0, 1 << 20, dtype=np.float32)
    x = np.concatenate([grid, gen.uniform(-126.0, 127.0, 1 << 18).astype(np.float32),
                        gen.uniform(-1.0, 1.0, 1 << 16).astype(np.float32),  # the reduced range itself
                        np.arange(-126, 128, dtype=np.float32),             # exact powers
                        np.arange(-126, 127, dtype=np.float32) + np.float32(0.5)])  # rounding ties of n
    y = attn.debug_exp2_poly(torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y - exact) / exact
    assert np.all(np.isfinite(y))
    assert rel.max() <= REL_BOUND, f"max relative error {rel.max():.3e} at x = {x[rel.argmax()]}"
    # 2^n exactly for integer n: p(0) = 1 and the exponent add is exact
    ints = np.arange(-126, 128, dtype=np.float32)
    yi = attn.debug_exp2_poly(torch.from_numpy(ints).cuda()).cpu().numpy()
    assert np.array_equal(yi, np.exp2(ints))


def test_exp2_poly_clamps_below_minus_126(attn):
    import torch
    x = np.array([-126.0, -126.5, -127.0, -150.0, -1e30, -np.inf, np.nan], dtype=np.float32)
    y = attn.debug_exp2_poly(torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.all(y == np.float32(2.0 ** -126)), y


def test_exp2_poly_odd_length_and_empty(attn):
    import torch
    x = np.array([0.0, 1.0, 2.5], dtype=np.float32)
    y = attn.debug_exp2_poly(torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y - np.exp2(x.astype(np.float64))) <= REL_BOUND * np.exp2(x.astype(np.float64)))
    assert attn.debug_exp2_poly(torch.empty(0, dtype=torch.float32, device="cuda")).numel() == 0


@pytest.mark.parametrize("B,H,Nq,Nk,D,causal", [
    (1, 2, 700, 900, 64, False),
    (1, 2, 700, 900, 64, True),
    (2, 1, 513, 640, 128, False),
    (1, 2, 640, 640, 128, True),
])
def test_forward_with_polynomial_exponentials_matches_the_oracle(attn, B, H, Nq, Nk, D, causal):
    import torch
    qn, kn, vn = synth.make_qkv(B, H, Nq, Nk, D, seed=90 + D + Nq, sigma_qk=2.0)
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    scale = 1.0 / math.sqrt(D)
    o, lse = attn.fwd_poly_exp(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    O, L = oracle.attn_full(qn, kn, vn, scale, causal)
    compare(o.cpu().numpy(), lse.cpu().numpy(), O, L, f"poly exp [{B},{H},{Nq},{Nk},{D}] causal={causal}")


def test_polynomial_forward_is_a_different_computation(attn):
    """The hook really routes exponentials through the polynomial: its P
    roundings differ from the exponential unit's somewhere in 16M weights."""
    import torch
    qn, kn, vn = synth.make_qkv(1, 4, 1024, 1024, 128, seed=95)
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    o1, l1 = attn.fwd(q, k, v)
    o2, l2 = attn.fwd_poly_exp(q, k, v)
    torch.cuda.synchronize()
    assert not (torch.equal(o1, o2) and torch.equal(l1, l2))
    assert (o1.float() - o2.float()).abs().max().item() <= 4e-3
