"""attn_fwd_host: the forward on host tensors with the copies in and out
overlapped over chunks of heads.  Its outputs must equal attn_fwd's bit for
bit (the same kernel on the same data), for any chunking, and match the
oracle."""
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


@pytest.mark.parametrize("B,H,Nq,Nk,D,causal,chunks", [
    (1, 8, 300, 257, 128, True, 3),     # uneven chunks, ragged tails
    (2, 3, 256, 512, 64, False, 8),     # more chunks than fit evenly
    (1, 2, 128, 128, 128, False, 64),   # more chunks than heads: capped at B*H
    (2, 4, 200, 200, 64, True, 0),      # default chunking
    (1, 1, 64, 1000, 128, False, 1),    # one chunk: plain copy, compute, copy
])
def test_host_entry_equals_device_entry(B, H, Nq, Nk, D, causal, chunks):
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    qn, kn, vn = synth.make_qkv(B, H, Nq, Nk, D, seed=5000 + Nq + chunks)
    scale = 1.0 / math.sqrt(D)
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (qn, kn, vn))
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        oh, lh = attn.fwd_host(qh, kh, vh, scale=scale, causal=causal, num_chunks=chunks)
    o1, l1 = attn.fwd(*(torch.from_numpy(x).cuda() for x in (qn, kn, vn)), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    assert torch.equal(oh, o1.cpu()) and torch.equal(lh, l1.cpu())
    O, L = oracle.attn_full(qn, kn, vn, scale, causal)
    compare(oh.numpy(), lh.numpy(), O, L, f"host entry [{B},{H},{Nq},{Nk},{D}] chunks={chunks}")


def test_host_entry_without_lse():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    qn, kn, vn = synth.make_qkv(1, 4, 160, 300, 64, seed=5100)
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (qn, kn, vn))
    oh, lh = attn.fwd_host(qh, kh, vh, causal=True, num_chunks=2, want_lse=False)
    assert lh is None
    o1, _ = attn.fwd(*(torch.from_numpy(x).cuda() for x in (qn, kn, vn)), causal=True)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    assert torch.equal(oh, o1.cpu())


@pytest.mark.parametrize("causal,chunks", [(False, 3), (True, 0)])
def test_fp8_host_entry_equals_device_entry(causal, chunks):
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    B, H, Nq, Nk = 1, 5, 200, 300
    q8, k8, v8 = synth.make_qkv_e4m3(B, H, Nq, Nk, 128, seed=5200 + chunks)
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (q8, k8, v8))
    qd, kd, vd = (torch.empty_like(x, device="cuda") for x in (qh, kh, vh))
    od = torch.empty((B, H, Nq, 128), dtype=torch.float16, device="cuda")
    ld = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.fp8_workspace_bytes(B, H, Nk, 128), dtype=torch.uint8, device="cuda")
    oh = torch.empty(od.shape, dtype=torch.float16).pin_memory()
    lh = torch.empty(ld.shape, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    code = attn.attn_fwd_fp8_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), lh.data_ptr(),
                                  qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), ld.data_ptr(),
                                  B, H, Nq, Nk, 128, 128 ** -0.5, causal, 0.5, 2.0, 1.5, ws.data_ptr(), ws.numel(),
                                  chunks, stream)
    assert code == attn.ATTN_OK
    torch.cuda.synchronize()
    o1, l1 = attn.fwd_fp8(*(torch.from_numpy(x).cuda() for x in (q8, k8, v8)), causal=causal,
                          q_descale=0.5, k_descale=2.0, v_descale=1.5)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    assert torch.equal(oh, o1.cpu()) and torch.equal(lh, l1.cpu())
