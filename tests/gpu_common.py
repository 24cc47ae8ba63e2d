"""Shared helpers of the GPU tests: run the CUDA path, compare with the oracle."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth

# Tolerances of the forward against the fp64 oracle (the same for every
# test): O max-abs error <= 4e-3 and relative RMS <= 1e-3, LSE max-abs <= 1e-3.
TOL_O_MAXABS = 4e-3
TOL_O_RELRMS = 1e-3
TOL_LSE_MAXABS = 1e-3


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def run_gpu(q, k, v, scale, causal):
    """Copy numpy fp16 inputs to the GPU, run the library, return numpy (o, lse)."""
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (q, k, v))
    o, lse = attn.fwd(tq, tk, tv, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    return o.cpu().numpy(), lse.cpu().numpy()


def compare(o_gpu, lse_gpu, O_ref, L_ref, label="", sigma_v=1.0):
    """Element-wise comparison; returns the three error figures.

    The O max-abs bound is stated for V of unit scale (every workload draws
    V from N(0, 1)); O is linear in V, so for V drawn with standard deviation
    sigma_v the bound is TOL_O_MAXABS * sigma_v.  The relative RMS bound is
    scale-free and the LSE does not depend on V."""
    o = o_gpu.astype(np.float64).reshape(O_ref.shape)
    l = lse_gpu.astype(np.float64).reshape(L_ref.shape)
    assert np.all(np.isfinite(o)), f"{label}: non-finite O"
    assert np.all(np.isfinite(l)), f"{label}: non-finite LSE"
    diff = o - O_ref
    max_abs = float(np.abs(diff).max())
    nrm = float(np.linalg.norm(O_ref))
    rel_rms = float(np.linalg.norm(diff) / nrm) if nrm > 0 else float(np.linalg.norm(diff))
    lse_err = float(np.abs(l - L_ref).max())
    assert max_abs <= TOL_O_MAXABS * sigma_v, f"{label}: O max-abs {max_abs:.3e}"
    assert rel_rms <= TOL_O_RELRMS, f"{label}: O rel-RMS {rel_rms:.3e}"
    assert lse_err <= TOL_LSE_MAXABS, f"{label}: LSE max-abs {lse_err:.3e}"
    return max_abs, rel_rms, lse_err


def full_parity(B, H, Nq, Nk, D, causal, seed, sigma_qk=1.0, sigma_v=1.0, scale=None):
    q, k, v = synth.make_qkv(B, H, Nq, Nk, D, seed, sigma_qk, sigma_v)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    o, lse = run_gpu(q, k, v, scale, causal)
    O, L = oracle.attn_full(q, k, v, scale, causal)
    return compare(o, lse, O, L, f"[{B},{H},{Nq},{Nk},{D}] causal={causal}", sigma_v=sigma_v)
