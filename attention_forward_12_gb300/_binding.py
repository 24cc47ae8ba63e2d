"""ctypes binding of ``libattn.so`` -- argument marshalling only.

Every step of the forward runs in the library's CUDA kernel; PyTorch is used
here only to allocate device memory and to name the current stream.  There
is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from ._build import LIB_PATH

ATTN_OK, ATTN_EINVAL, ATTN_EUNSUPPORTED, ATTN_ECUDA, ATTN_ETIMEOUT, ATTN_ESCRATCH, ATTN_ETOOLONG = range(7)
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
MAX_KEYS_PER_PASS = 1 << 19

# Every symbol the C header declares; the CPU tests check they are exported.
EXPORTS = ("attn_fwd", "attn_fwd_launch_count", "attn_fwd_host", "attn_fwd_splitkv", "attn_splitkv_workspace_bytes", "attn_splitkv_suggest",
           "attn_fwd_splitkv_noalloc", "attn_fwd_fp8", "attn_fwd_fp8_host", "attn_fp8_workspace_bytes", "attn_debug_pack_e4m3",
           "attn_debug_exp2_poly", "attn_debug_fwd_poly_exp", "attn_strerror", "attn_get_status", "attn_debug_set",
           "attn_version")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (code {code})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it with "
                    "attention_forward_12_gb300.build() (nvcc, sm_103a)")
            lib = ctypes.CDLL(path)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            lib.attn_fwd.restype = i32
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     ctypes.c_float, i32, vp]
            lib.attn_fwd_launch_count.restype = i32
            lib.attn_fwd_launch_count.argtypes = [i32] * 6
            lib.attn_fwd_host.restype = i32
            lib.attn_fwd_host.argtypes = [vp] * 10 + [i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, vp]
            lib.attn_fwd_splitkv.restype = i32
            lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                             ctypes.c_float, i32, i32, vp, ctypes.c_size_t, vp]
            lib.attn_fwd_splitkv_noalloc.restype = i32
            lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                     ctypes.c_float, i32, i32, vp]
            f32 = ctypes.c_float
            lib.attn_fwd_fp8.restype = i32
            lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, f32, f32, f32,
                                         vp, ctypes.c_size_t, vp]
            lib.attn_fwd_fp8_host.restype = i32
            lib.attn_fwd_fp8_host.argtypes = [vp] * 10 + [i32, i32, i32, i32, i32, f32, i32, f32, f32, f32, vp,
                                                          ctypes.c_size_t, i32, vp]
            lib.attn_fp8_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_fp8_workspace_bytes.argtypes = [i32, i32, i32, i32]
            lib.attn_debug_pack_e4m3.restype = i32
            lib.attn_debug_pack_e4m3.argtypes = [vp, vp, i32, vp]
            lib.attn_debug_exp2_poly.restype = i32
            lib.attn_debug_exp2_poly.argtypes = [vp, vp, i32, vp]
            lib.attn_debug_fwd_poly_exp.restype = i32
            lib.attn_debug_fwd_poly_exp.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                    ctypes.c_float, i32, vp]
            lib.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_splitkv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.attn_splitkv_suggest.restype = i32
            lib.attn_splitkv_suggest.argtypes = [i32, i32, i32, i32, i32, i32]
            lib.attn_strerror.restype = ctypes.c_char_p
            lib.attn_strerror.argtypes = [i32]
            lib.attn_get_status.restype = i32
            lib.attn_get_status.argtypes = [vp]
            lib.attn_debug_set.restype = i32
            lib.attn_debug_set.argtypes = [ctypes.c_ulonglong, i32]
            lib.attn_version.restype = i32
            lib.attn_version.argtypes = []
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load_library().attn_strerror(int(code)).decode()


def attn_fwd(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None,
             B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
             stream: int | None) -> int:
    """Direct call of the C entry point with raw device pointers; returns the code."""
    return load_library().attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H),
                                   int(Nq), int(Nk), int(D), float(scale), int(bool(causal)),
                                   stream)


def fwd_launch_count(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool) -> int:
    """Kernels attn_fwd enqueues for these sizes on the current device (1 or 2)."""
    return int(load_library().attn_fwd_launch_count(int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal))))


def attn_fwd_host(qh: int, kh: int, vh: int, oh: int, lh: int | None, qd: int, kd: int, vd: int, od: int,
                  ld: int | None, B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
                  num_chunks: int, stream: int | None) -> int:
    """Direct call of the host-buffer entry point (raw host and device pointers)."""
    return load_library().attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, int(B), int(H), int(Nq), int(Nk),
                                        int(D), float(scale), int(bool(causal)), int(num_chunks), stream)


def attn_fwd_splitkv(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None,
                     B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
                     num_splits: int, ws_ptr: int | None, ws_bytes: int, stream: int | None) -> int:
    """Direct call of the split-KV entry point with raw device pointers."""
    return load_library().attn_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(Nq),
                                           int(Nk), int(D), float(scale), int(bool(causal)),
                                           int(num_splits), ws_ptr, int(ws_bytes), stream)


def attn_fwd_splitkv_noalloc(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None,
                             B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
                             num_splits: int, stream: int | None) -> int:
    """Split-KV forward that allocates nothing: its scratch is a buffer built
    into the library (see attn.h for the limit and the sharing rules)."""
    return load_library().attn_fwd_splitkv_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H),
                                                   int(Nq), int(Nk), int(D), float(scale),
                                                   int(bool(causal)), int(num_splits), stream)


def attn_fwd_fp8(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None,
                 B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
                 q_descale: float, k_descale: float, v_descale: float,
                 ws_ptr: int | None, ws_bytes: int, stream: int | None) -> int:
    """Direct call of the E4M3 entry point with raw device pointers."""
    return load_library().attn_fwd_fp8(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(Nq), int(Nk),
                                       int(D), float(scale), int(bool(causal)), float(q_descale),
                                       float(k_descale), float(v_descale), ws_ptr, int(ws_bytes), stream)


def attn_fwd_fp8_host(qh: int, kh: int, vh: int, oh: int, lh: int | None, qd: int, kd: int, vd: int, od: int,
                      ld: int | None, B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
                      q_descale: float, k_descale: float, v_descale: float, ws_ptr: int | None, ws_bytes: int,
                      num_chunks: int, stream: int | None) -> int:
    """Direct call of the E4M3 host-buffer entry point (raw pointers)."""
    return load_library().attn_fwd_fp8_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, int(B), int(H), int(Nq), int(Nk),
                                            int(D), float(scale), int(bool(causal)), float(q_descale),
                                            float(k_descale), float(v_descale), ws_ptr, int(ws_bytes),
                                            int(num_chunks), stream)


def fp8_workspace_bytes(B: int, H: int, Nk: int, D: int) -> int:
    return int(load_library().attn_fp8_workspace_bytes(int(B), int(H), int(Nk), int(D)))


def splitkv_workspace_bytes(B: int, H: int, Nq: int, D: int, num_splits: int) -> int:
    return int(load_library().attn_splitkv_workspace_bytes(int(B), int(H), int(Nq), int(D), int(num_splits)))


def splitkv_suggest(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool) -> int:
    return int(load_library().attn_splitkv_suggest(int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal))))


def _current_stream_ptr(device) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def fwd(q, k, v, scale: float | None = None, causal: bool = False, out=None, lse=None,
        want_lse: bool = True, _entry=None):
    """O = softmax(scale * Q K^T) V on the GPU; returns (o, lse).

    q: fp16 CUDA tensor [B,H,Nq,D], k and v: [B,H,Nk,D], contiguous.
    scale defaults to 1/sqrt(D).  out / lse may be preallocated
    ([B,H,Nq,D] fp16 and [B,H,Nq] fp32).  Runs on the current stream.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float16):
            raise TypeError(f"{name} must be a CUDA float16 tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D [B,H,N,D] tensor")
    B, H, Nq, D = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("k and v must be [B,H,Nk,D] with q's B, H and D")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    entry = attn_fwd if _entry is None else _entry
    code = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                 lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, D, scale, causal,
                 _current_stream_ptr(q.device))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd")
    return out, lse


def attn_debug_fwd_poly_exp(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None,
                            B: int, H: int, Nq: int, Nk: int, D: int, scale: float, causal: bool,
                            stream: int | None) -> int:
    """The testing hook that runs attn_fwd with a quarter of the exponentials
    on the FMA-pipe polynomial (raw device pointers; returns the code)."""
    return load_library().attn_debug_fwd_poly_exp(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H),
                                                  int(Nq), int(Nk), int(D), float(scale),
                                                  int(bool(causal)), stream)


def fwd_poly_exp(q, k, v, scale: float | None = None, causal: bool = False):
    """fwd through the polynomial-exponential testing hook; returns (o, lse)."""
    return fwd(q, k, v, scale=scale, causal=causal, _entry=attn_debug_fwd_poly_exp)


def fwd_host(q, k, v, scale: float | None = None, causal: bool = False, num_chunks: int = 0,
             device=None, dev_buffers=None, out=None, lse=None, want_lse: bool = True):
    """attn_fwd on CPU tensors (pinned for overlap); returns host (o, lse).

    q, k, v: contiguous CPU float16 tensors [B,H,N,D].  dev_buffers: an
    optional (q, k, v, o, lse) tuple of CUDA tensors of the full sizes,
    allocated here when not given.  The call synchronises the current
    stream before returning, so the host outputs are ready."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (isinstance(t, torch.Tensor) and not t.is_cuda and t.dtype == torch.float16):
            raise TypeError(f"{name} must be a CPU float16 tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D [B,H,N,D] tensor")
    B, H, Nq, D = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("k and v must be [B,H,Nk,D] with q's B, H and D")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev_buffers is None:
        dev_buffers = (torch.empty_like(q, device=device), torch.empty_like(k, device=device),
                       torch.empty_like(v, device=device), torch.empty_like(q, device=device),
                       torch.empty((B, H, Nq), dtype=torch.float32, device=device) if want_lse else None)
    qd, kd, vd, od, ld = dev_buffers
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32)
    stream = _current_stream_ptr(device)
    code = attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if want_lse else None, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                         od.data_ptr(), ld.data_ptr() if want_lse else None, B, H, Nq, Nk, D, scale, causal,
                         num_chunks, stream)
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_host")
    torch.cuda.current_stream(device).synchronize()
    return out, (lse if want_lse else None)


def fwd_splitkv(q, k, v, scale: float | None = None, causal: bool = False, num_splits: int | None = None,
                workspace=None, out=None, lse=None, want_lse: bool = True):
    """Split-KV forward (see attn.h); returns (o, lse).  num_splits defaults
    to the library's suggestion; the workspace is allocated with torch when
    not given (a uint8 CUDA tensor of at least splitkv_workspace_bytes)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float16):
            raise TypeError(f"{name} must be a CUDA float16 tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D [B,H,N,D] tensor")
    B, H, Nq, D = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("k and v must be [B,H,Nk,D] with q's B, H and D")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if num_splits is None:
        num_splits = max(1, splitkv_suggest(B, H, Nq, Nk, D, causal))
    need = splitkv_workspace_bytes(B, H, Nq, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    code = attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, D, scale, causal,
                            num_splits, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _current_stream_ptr(q.device))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_splitkv")
    return out, lse


def fwd_fp8(q, k, v, scale: float | None = None, causal: bool = False, q_descale: float = 1.0,
            k_descale: float = 1.0, v_descale: float = 1.0, workspace=None, out=None, lse=None,
            want_lse: bool = True):
    """Forward on E4M3 inputs (see attn.h); returns (o, lse), o fp16.

    q, k, v: contiguous CUDA tensors [B,H,N,128] of one byte per element
    (torch.float8_e4m3fn, or uint8 holding E4M3 bit patterns).  The
    workspace (V transposed) is allocated with torch when not given."""
    import torch
    byte_types = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype in byte_types):
            raise TypeError(f"{name} must be a CUDA float8_e4m3fn (or uint8) tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D [B,H,N,D] tensor")
    B, H, Nq, D = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("k and v must be [B,H,Nk,D] with q's B, H and D")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = fp8_workspace_bytes(B, H, Nk, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, H, Nq, D), dtype=torch.float16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    code = attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, D, scale, causal,
                        q_descale, k_descale, v_descale, workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _current_stream_ptr(q.device))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_fp8")
    return out, lse


def debug_pack_e4m3(x):
    """The FP8 forward's E4M3 rounding of P applied to a float32 CUDA tensor
    (numel a multiple of 4); returns the E4M3 bytes as a uint8 tensor."""
    import torch
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise TypeError("x must be a contiguous CUDA float32 tensor")
    if x.numel() % 4:
        raise ValueError("numel must be a multiple of 4")
    out = torch.empty(x.numel() // 4, dtype=torch.int32, device=x.device)
    code = load_library().attn_debug_pack_e4m3(x.data_ptr(), out.data_ptr(), x.numel() // 4,
                                               _current_stream_ptr(x.device))
    if code != ATTN_OK:
        raise AttnError(code, "attn_debug_pack_e4m3")
    return out.view(torch.uint8)


def debug_exp2_poly(x):
    """2^x by the forward's FMA-pipe polynomial, for a contiguous float32
    CUDA tensor; returns a new tensor."""
    import torch
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise TypeError("x must be a contiguous CUDA float32 tensor")
    out = torch.empty_like(x)
    code = load_library().attn_debug_exp2_poly(x.data_ptr(), out.data_ptr(), x.numel(),
                                               _current_stream_ptr(x.device))
    if code != ATTN_OK:
        raise AttnError(code, "attn_debug_exp2_poly")
    return out


def get_status(stream: int | None = None) -> int:
    """Synchronise the stream and read-and-clear the device status word."""
    if stream is None:
        stream = _current_stream_ptr(None)
    return load_library().attn_get_status(stream)


def debug_set(wait_timeout_ns: int = 2_000_000_000, drop_kv_tile: int = -1) -> int:
    return load_library().attn_debug_set(int(wait_timeout_ns), int(drop_kv_tile))


def version() -> int:
    return load_library().attn_version()
