"""Failure detection on the GPU without a fault: one TMA load is never
issued (attn_debug_set's drop_kv_tile), so the wait for it runs out after a
short limit; the kernel must stop cleanly, report ATTN_ETIMEOUT through
attn_get_status, and leave the context usable for the next correct call."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from gpu_common import compare, torch_cuda

pytestmark = pytest.mark.gpu


def test_dropped_load_times_out_and_context_survives():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    B, H, N, D = 1, 2, 512, 128
    qn, kn, vn = synth.make_qkv(B, H, N, N, D, seed=21)
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    assert attn.get_status() == attn.ATTN_OK
    try:
        assert attn.debug_set(50_000_000, 1) == attn.ATTN_OK  # 50 ms limit, key tile 1 never loaded
        attn.fwd(q, k, v, causal=False)
        torch.cuda.synchronize()
        assert attn.get_status() == attn.ATTN_ETIMEOUT
        assert attn.get_status() == attn.ATTN_OK  # read-and-clear
    finally:
        attn.debug_set(2_000_000_000, -1)
    o, lse = attn.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    O, L = oracle.attn_full(qn, kn, vn, 1.0 / math.sqrt(D), False)
    compare(o.cpu().numpy(), lse.cpu().numpy(), O, L, "after timeout")
