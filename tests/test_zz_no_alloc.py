"""attn_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory (a serving loop that must stay out of the allocator,
a plugin whose host owns all device memory).  Its scratch is a buffer built
into the library, shared by every call and keeping the last call's
contents, so the test makes two calls in a row on different problems and
checks each against the existing split-KV entry point (which uses a
caller-provided workspace), within the tolerances of the other GPU tests,
and against the fp64 oracle.  Around the second call the device's free
memory and torch's reserved memory must not move: the entry point allocates
nothing.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from gpu_common import compare, torch_cuda

pytestmark = pytest.mark.gpu


def _noalloc_call(attn, lib, q, k, v, o, lse, scale, causal, splits):
    import torch
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.attn_fwd_splitkv_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                      ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                      ctypes.c_void_p(lse.data_ptr()), B, H, Nq, Nk, D,
                                      ctypes.c_float(scale), int(causal), splits,
                                      ctypes.c_void_p(stream))
    assert rc == attn.ATTN_OK, attn.strerror(rc)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    lib = attn.load_library()
    problems = [
        # B, H, Nq, Nk, D, causal, splits, seed
        (1, 8, 128, 8192, 128, False, 12, 71),
        (2, 2, 300, 2000, 64, True, 5, 72),   # smaller: stale parts of call 1 must not leak in
    ]
    for n, (B, H, Nq, Nk, D, causal, splits, seed) in enumerate(problems):
        qn, kn, vn = synth.make_qkv(B, H, Nq, Nk, D, seed)
        q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
        scale = 1.0 / math.sqrt(D)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        torch.cuda.synchronize()
        free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
        _noalloc_call(attn, lib, q, k, v, o, lse, scale, causal, splits)
        torch.cuda.synchronize()
        free1, reserved1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
        if n > 0:  # the first call may load the library's kernels; the second allocates nothing
            assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
            assert reserved1 == reserved0
        o_ref, lse_ref = attn.fwd_splitkv(q, k, v, scale=scale, causal=causal, num_splits=splits)
        torch.cuda.synchronize()
        assert attn.get_status() == attn.ATTN_OK
        label = f"no-alloc [{B},{H},{Nq},{Nk},{D}]"
        og, lg = o.cpu().numpy(), lse.cpu().numpy()
        compare(og, lg, o_ref.cpu().numpy().astype(np.float64), lse_ref.cpu().numpy().astype(np.float64), label)
        O, L = oracle.attn_full(qn, kn, vn, scale, causal)
        compare(og, lg, O, L, label + " vs oracle")


def test_noalloc_rejects_problems_beyond_its_scratch():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    lib = attn.load_library()
    q = torch.zeros(1, 64, 16384, 128, dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    # 8 shares * 64 heads * 16384 rows * 129 floats is far beyond the built-in
    # scratch: rejected on the host, nothing is enqueued
    rc = lib.attn_fwd_splitkv_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                      None, 1, 64, 16384, 16384, 128, ctypes.c_float(0.1), 0, 8, None)
    assert rc == attn.ATTN_ESCRATCH
