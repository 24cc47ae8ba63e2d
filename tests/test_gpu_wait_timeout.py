"""Failure detection on the GPU without a fault: one TMA load is never
issued (attn_debug_set's drop_kv_tile), so the wait for it runs out after a
short limit; the kernel must stop cleanly, report ATTN_ETIMEOUT through
attn_get_status -- and, until that report is read, through every call, at
once and without a device synchronisation -- and leave the context usable
for the next correct call."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from gpu_common import compare, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_dropped_load_times_out_and_context_survives(D):
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    B, H, N = 1, 2, 512
    qn, kn, vn = synth.make_qkv(B, H, N, N, D, seed=21)
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    assert attn.get_status() == attn.ATTN_OK
    try:
        assert attn.debug_set(50_000_000, 1) == attn.ATTN_OK  # 50 ms limit, key tile 1 never loaded
        attn.fwd(q, k, v, causal=False)
        torch.cuda.synchronize()
    finally:
        attn.debug_set(2_000_000_000, -1)
    # The error is pending: every entry point refuses to enqueue, without a sync.
    for call in (lambda: attn.fwd(q, k, v, causal=False),
                 lambda: attn.fwd_splitkv(q, k, v, num_splits=2)):
        with pytest.raises(attn.AttnError) as e:
            call()
        assert e.value.code == attn.ATTN_ETIMEOUT
    assert attn.get_status() == attn.ATTN_ETIMEOUT
    assert attn.get_status() == attn.ATTN_OK  # read-and-clear
    o, lse = attn.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    O, L = oracle.attn_full(qn, kn, vn, 1.0 / math.sqrt(D), False)
    compare(o.cpu().numpy(), lse.cpu().numpy(), O, L, "after timeout")


def test_dropped_load_times_out_in_the_e4m3_forward():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    q8, k8, v8 = synth.make_qkv_e4m3(1, 2, 512, 512, 128, seed=22)
    q, k, v = (torch.from_numpy(x).cuda() for x in (q8, k8, v8))
    assert attn.get_status() == attn.ATTN_OK
    try:
        assert attn.debug_set(50_000_000, 1) == attn.ATTN_OK
        attn.fwd_fp8(q, k, v)
        torch.cuda.synchronize()
        assert attn.get_status() == attn.ATTN_ETIMEOUT
    finally:
        attn.debug_set(2_000_000_000, -1)
    o, lse = attn.fwd_fp8(q, k, v)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    O, L = oracle.attn_full_e4m3(q8, k8, v8, 128 ** -0.5, False)
    og = o.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(og - O) / np.linalg.norm(O) <= 0.05
    assert np.abs(lse.cpu().numpy() - L).max() <= 1e-3


def test_dropped_load_times_out_in_the_host_entry():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    qn, kn, vn = synth.make_qkv(1, 4, 256, 256, 64, seed=23)
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (qn, kn, vn))
    assert attn.get_status() == attn.ATTN_OK
    try:
        assert attn.debug_set(50_000_000, 1) == attn.ATTN_OK
        attn.fwd_host(qh, kh, vh, num_chunks=2)
        assert attn.get_status() == attn.ATTN_ETIMEOUT
    finally:
        attn.debug_set(2_000_000_000, -1)
    oh, lh = attn.fwd_host(qh, kh, vh, num_chunks=2)
    assert attn.get_status() == attn.ATTN_OK
    O, L = oracle.attn_full(qn, kn, vn, 1.0 / math.sqrt(64), False)
    compare(oh.numpy(), lh.numpy(), O, L, "host entry after timeout")
