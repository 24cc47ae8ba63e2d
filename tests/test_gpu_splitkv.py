"""Split-KV forward (keys of each query tile divided into shares computed by
separate CTAs, then merged with the carrier merge): element-wise parity with
the fp64 oracle, agreement with the single-pass forward, and the decode-like
shapes it exists for, including shares that hold no admissible key."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from gpu_common import compare, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    attn.load_library()


def _run(qn, kn, vn, scale, causal, splits):
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    o, lse = attn.fwd_splitkv(q, k, v, scale=scale, causal=causal, num_splits=splits)
    o1, l1 = attn.fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    return o.cpu().numpy(), lse.cpu().numpy(), o1.cpu().numpy(), l1.cpu().numpy()


CASES = [
    # B, H, Nq, Nk, D, causal, splits
    (1, 8, 1, 4097, 128, False, 16),      # one query row, long keys (decode)
    (2, 4, 64, 8192, 64, False, 8),
    (1, 2, 130, 5000, 128, True, 4),      # causal: shares past the diagonal are empty
    (1, 1, 300, 300, 128, True, 3),
    (1, 3, 200, 1000, 64, False, 1),      # one share
    (1, 2, 128, 512, 128, False, 9),      # more shares than key tiles: empty shares
    (2, 2, 700, 900, 64, True, 5),
    # one key tile per share, the diagonal tile alone in the last one
    (1, 1, 256, 256, 64, True, 4),
    (1, 2, 256, 256, 128, True, 4),
]


@pytest.mark.parametrize("B,H,Nq,Nk,D,causal,splits", CASES)
def test_splitkv_matches_oracle_and_single_pass(B, H, Nq, Nk, D, causal, splits):
    qn, kn, vn = synth.make_qkv(B, H, Nq, Nk, D, seed=3000 + Nq + Nk + splits)
    scale = 1.0 / math.sqrt(D)
    o, lse, o1, l1 = _run(qn, kn, vn, scale, causal, splits)
    O, L = oracle.attn_full(qn, kn, vn, scale, causal)
    compare(o, lse, O, L, f"split-KV x{splits}")
    compare(o, lse, o1.astype(np.float64), l1.astype(np.float64), "split-KV vs single pass")


def test_splitkv_peaked_long():
    qn, kn, vn = synth.make_qkv(1, 4, 256, 16384, 128, seed=31, sigma_qk=3.0)
    scale = 1.0 / math.sqrt(128)
    o, lse, _, _ = _run(qn, kn, vn, scale, False, 24)
    O, L = oracle.attn_full(qn, kn, vn, scale, False)
    compare(o, lse, O, L, "split-KV peaked")


def test_splitkv_suggest_fills_the_gpu():
    torch_cuda()
    import attention_forward_12_gb300 as attn
    s = attn.splitkv_suggest(1, 8, 1, 32768, 128, False)
    assert 2 <= s <= 256
    assert attn.splitkv_suggest(4, 32, 16384, 16384, 128, False) == 1


def test_share_suggestion_follows_the_measured_cost():
    """The suggested share count splits decode-like shapes (few CTAs, many
    keys) and leaves shapes whose grid already fills the SMs to the single
    pass (the split-KV path then only adds the parts and the merge)."""
    torch_cuda()
    import attention_forward_12_gb300 as attn
    assert attn.splitkv_suggest(1, 8, 4096, 4096, 64, False) == 1      # 128 CTAs
    assert attn.splitkv_suggest(1, 16, 8192, 8192, 128, False) == 1    # 512 CTAs
    assert attn.splitkv_suggest(1, 8, 128, 32768, 128, False) >= 8     # 8 CTAs, 256 key tiles
    assert attn.splitkv_suggest(4, 8, 1, 65536, 128, False) >= 4       # 32 CTAs, 512 key tiles
    # 2^20 keys: never a share longer than one pass may accumulate
    s = attn.splitkv_suggest(1, 1, 3, 1 << 20, 64, False)
    assert s >= 2 and (8192 + s - 1) // s * 128 <= attn.MAX_KEYS_PER_PASS
