"""GB300-native (sm_103a) fused scaled-dot-product attention forward.

``fwd(q, k, v, scale, causal) -> (o, lse)`` runs the hand-written tcgen05 /
TMA kernel of ``csrc/attn_fwd.cu`` through its C ABI (``include/attn.h``).
``build()`` compiles that library in place with nvcc.
"""
from ._binding import (ATTN_ECUDA, ATTN_EINVAL, ATTN_ESCRATCH, ATTN_ETIMEOUT, ATTN_ETOOLONG, ATTN_EUNSUPPORTED,
                       ATTN_OK, EXPORTS, MAX_KEYS_PER_PASS, NOALLOC_SCRATCH_BYTES, AttnError,
                       attn_debug_fwd_poly_exp, attn_fwd, attn_fwd_fp8, attn_fwd_fp8_host, attn_fwd_host,
                       attn_fwd_splitkv, attn_fwd_splitkv_noalloc, debug_exp2_poly, debug_pack_e4m3, debug_set,
                       fp8_workspace_bytes, fwd, fwd_fp8, fwd_host, fwd_launch_count, fwd_poly_exp, fwd_splitkv,
                       get_status, load_library, splitkv_suggest, splitkv_workspace_bytes, strerror,
                       version)
from ._build import LIB_PATH, build

__all__ = ["fwd", "attn_fwd", "fwd_launch_count", "fwd_host", "attn_fwd_host", "attn_fwd_fp8_host", "fwd_fp8", "attn_fwd_fp8",
           "fp8_workspace_bytes", "debug_pack_e4m3", "debug_exp2_poly", "fwd_poly_exp", "attn_debug_fwd_poly_exp",
           "fwd_splitkv", "attn_fwd_splitkv", "attn_fwd_splitkv_noalloc",
           "NOALLOC_SCRATCH_BYTES", "MAX_KEYS_PER_PASS", "ATTN_ESCRATCH", "ATTN_ETOOLONG", "splitkv_suggest",
           "splitkv_workspace_bytes", "get_status", "debug_set", "strerror", "version", "build",
           "load_library", "LIB_PATH", "EXPORTS", "AttnError", "ATTN_OK", "ATTN_EINVAL",
           "ATTN_EUNSUPPORTED", "ATTN_ECUDA", "ATTN_ETIMEOUT"]
