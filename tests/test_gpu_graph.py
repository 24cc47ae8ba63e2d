"""The forward entry points are asynchronous, allocate nothing and never
synchronise the host, so they can be captured in a CUDA graph: a captured
call replayed on new inputs (copied into the captured buffers) gives the
same bytes as a direct call."""
import math

import pytest

from attention_forward_12_gb300 import synth
from gpu_common import torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,causal,B,H,N", [(64, False, 1, 4, 384), (128, True, 1, 4, 384),
                                           (64, False, 1, 16, 8192)])  # pairs, then a dependent single-tile launch
def test_forward_replays_from_a_cuda_graph(D, causal, B, H, N):
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    if N == 8192:
        assert attn.fwd_launch_count(B, H, N, N, D, causal) == 2
    bufs = [torch.from_numpy(x).cuda() for x in synth.make_qkv(B, H, N, N, D, seed=31)]
    o = torch.empty_like(bufs[0])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    attn.fwd(*bufs, causal=causal, out=o, lse=lse)  # first call on the device before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            attn.fwd(*bufs, causal=causal, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    for seed in (32, 33):  # new inputs into the captured buffers, replay, compare with a direct call
        new = [torch.from_numpy(x).cuda() for x in synth.make_qkv(B, H, N, N, D, seed=seed)]
        for b, n in zip(bufs, new):
            b.copy_(n)
        g.replay()
        o_ref, l_ref = attn.fwd(*new, causal=causal)
        torch.cuda.synchronize()
        assert attn.get_status() == attn.ATTN_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_fp8_forward_replays_from_a_cuda_graph():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    B, H, N = 1, 2, 300
    bufs = [torch.from_numpy(x).cuda() for x in synth.make_qkv_e4m3(B, H, N, N, 128, seed=34)]
    ws = torch.empty(attn.fp8_workspace_bytes(B, H, N, 128), dtype=torch.uint8, device="cuda")
    o = torch.empty((B, H, N, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    attn.fwd_fp8(*bufs, workspace=ws, out=o, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            attn.fwd_fp8(*bufs, workspace=ws, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    new = [torch.from_numpy(x).cuda() for x in synth.make_qkv_e4m3(B, H, N, N, 128, seed=35)]
    for b, n in zip(bufs, new):
        b.copy_(n)
    g.replay()
    o_ref, l_ref = attn.fwd_fp8(*new)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
