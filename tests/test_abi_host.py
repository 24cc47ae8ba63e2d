"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every symbol include/attn.h declares, and rejects bad arguments
before touching the device."""
import os
import re

import pytest

import attention_forward_12_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    attn.build()
    return attn.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_and_binding_agree(lib):
    decl = declared_functions()
    assert decl, "no declarations parsed from include/attn.h"
    assert sorted(attn.EXPORTS) == decl


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_strerror(lib):
    assert attn.version() == 4
    for code in (attn.ATTN_OK, attn.ATTN_EINVAL, attn.ATTN_EUNSUPPORTED, attn.ATTN_ECUDA,
                 attn.ATTN_ETIMEOUT, attn.ATTN_ESCRATCH, attn.ATTN_ETOOLONG, 99):
        assert isinstance(attn.strerror(code), str) and attn.strerror(code)
    assert "splitkv" in attn.strerror(attn.ATTN_ETOOLONG)
    assert attn.strerror(attn.ATTN_ETOOLONG) != attn.strerror(99)


def test_header_constants_match_binding(lib):
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    assert int(re.search(r"#define ATTN_MAX_KEYS_PER_PASS (\d+)", text).group(1)) == attn.MAX_KEYS_PER_PASS
    assert int(re.search(r"ATTN_ETOOLONG = (\d+)", text).group(1)) == attn.ATTN_ETOOLONG


A = 1 << 20  # a 16-byte aligned fake address: validation never dereferences it


@pytest.mark.parametrize("args,code", [
    ((0, A, A, 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0), attn.ATTN_EINVAL),      # null q
    ((A, A, A, 0, None, 1, 1, 8, 8, 64, 0.1, 0), attn.ATTN_EINVAL),          # null o
    ((A, A, A, 2 * A, None, -1, 1, 8, 8, 64, 0.1, 0), attn.ATTN_EINVAL),     # negative B
    ((A, A, A, 2 * A, None, 1, 1, 8, 0, 64, 0.1, 0), attn.ATTN_EINVAL),      # Nk = 0
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 64, -0.5, 0), attn.ATTN_EINVAL),     # negative scale
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 64, float("nan"), 0), attn.ATTN_EINVAL),
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 96, 0.1, 0), attn.ATTN_EUNSUPPORTED),  # D
    ((A + 2, A, A, 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0), attn.ATTN_EUNSUPPORTED),  # misaligned q
    ((A, A, A, 2 * A, A + 2, 1, 1, 8, 8, 64, 0.1, 0), attn.ATTN_EUNSUPPORTED),  # misaligned lse
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0.1, 0), attn.ATTN_EUNSUPPORTED),    # o overlaps q
    ((A, A, A, 2 * A, None, 300, 300, 8, 8, 64, 0.1, 0), attn.ATTN_EUNSUPPORTED),  # B*H > 65535
    ((A, A, A, 2 * A, None, 0, 4, 8, 8, 64, 0.1, 0), attn.ATTN_OK),          # empty: no-op
    ((A, A, A, 2 * A, None, 2, 4, 0, 8, 64, 0.1, 1), attn.ATTN_OK),          # Nq = 0: no-op
])
def test_argument_validation_without_device(lib, args, code):
    assert attn.attn_fwd(*args, None) == code


FAR = 1 << 40  # an output address far from the fake inputs, so no overlap is reported
LONG = (1 << 19) + 1  # one key more than a single pass may accumulate per row


@pytest.mark.parametrize("Nq,Nk,causal,code", [
    (8, LONG, 0, attn.ATTN_ETOOLONG),      # non-causal: every row accumulates Nk keys
    (LONG, LONG, 1, attn.ATTN_ETOOLONG),   # causal: the last row accumulates min(Nk, Nq) keys
])
def test_key_range_beyond_one_pass_is_rejected_without_device(lib, Nq, Nk, causal, code):
    assert attn.attn_fwd(A, A, A, FAR, None, 1, 1, Nq, Nk, 64, 0.1, causal, None) == code
    assert attn.attn_debug_fwd_poly_exp(A, A, A, FAR, None, 1, 1, Nq, Nk, 64, 0.1, causal, None) == code


def test_split_kv_share_beyond_one_pass_is_rejected_without_device(lib):
    W2 = 1 << 44  # workspace far from everything
    nk = 2 * (1 << 19) + 128  # 8193 key tiles: two shares hold 4097 tiles, one more than a pass
    f = attn.attn_fwd_splitkv
    assert f(A, A, A, FAR, None, 1, 1, 8, nk, 64, 0.1, 0, 2, W2, 1 << 30, None) == attn.ATTN_ETOOLONG
    g = attn.attn_fwd_splitkv_noalloc
    assert g(A, A, A, FAR, None, 1, 1, 8, nk, 64, 0.1, 0, 2, None) == attn.ATTN_ETOOLONG


def test_debug_hook_validation(lib):
    assert attn.debug_set(0, -1) == attn.ATTN_EINVAL
    assert attn.debug_set(10, -2) == attn.ATTN_EINVAL
    assert attn.debug_set(2_000_000_000, -1) == attn.ATTN_OK


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 4, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        attn.fwd(x, x, x)


def test_missing_library_fails_loudly(tmp_path):
    from attention_forward_12_gb300 import _binding
    saved = _binding._lib
    _binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            _binding.load_library(str(tmp_path / "nope.so"))
    finally:
        _binding._lib = saved


def test_splitkv_workspace_bytes(lib):
    assert attn.splitkv_workspace_bytes(2, 3, 100, 128, 4) == 4 * 2 * 3 * 100 * 129 * 4
    assert attn.splitkv_workspace_bytes(1, 1, 1, 64, 1) == 65 * 4
    for bad in [(1, 1, 1, 96, 2), (1, 1, 1, 64, 0), (1, 1, 1, 64, 257), (-1, 1, 1, 64, 2)]:
        assert attn.splitkv_workspace_bytes(*bad) == 0
    assert attn.splitkv_suggest(1, 1, 1, 1, 96, 0) == 0


W = 1 << 24  # fake 16-byte aligned workspace address, far from A


@pytest.mark.parametrize("splits,ws,nbytes,code", [
    (0, W, 1 << 20, attn.ATTN_EINVAL),           # too few shares
    (257, W, 1 << 20, attn.ATTN_EINVAL),         # too many shares
    (2, 0, 1 << 20, attn.ATTN_EINVAL),           # no workspace
    (2, W, 100, attn.ATTN_EINVAL),               # workspace too small
    (2, W + 4, 1 << 20, attn.ATTN_EUNSUPPORTED),  # misaligned workspace
    (2, A, 1 << 20, attn.ATTN_EUNSUPPORTED),     # workspace overlaps q
])
def test_splitkv_validation_without_device(lib, splits, ws, nbytes, code):
    assert attn.attn_fwd_splitkv(A, A, A, 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, splits, ws, nbytes, None) == code


def test_noalloc_rejects_before_touching_the_device(lib):
    f = attn.attn_fwd_splitkv_noalloc
    assert f(A, A, A, 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, 0, None) == attn.ATTN_EINVAL
    assert f(A, A, A, 2 * A, None, 1, 1, 8, 8, 96, 0.1, 0, 2, None) == attn.ATTN_EUNSUPPORTED
    # 8 * 64 * 16384 * 129 * 4 bytes of parts: larger than the built-in scratch
    far = 1 << 40  # an output address far from the fake inputs, so no overlap is reported
    assert f(A, A, A, far, None, 1, 64, 16384, 4096, 128, 0.1, 0, 8, None) == attn.ATTN_ESCRATCH
    assert "scratch" in attn.strerror(attn.ATTN_ESCRATCH)
    assert f(A, A, A, 2 * A, None, 0, 4, 8, 8, 64, 0.1, 0, 2, None) == attn.ATTN_OK  # empty problem


def test_fp8_workspace_bytes(lib):
    assert attn.fp8_workspace_bytes(2, 3, 100, 128) == 2 * 3 * 128 * 112  # rows rounded up to 16 keys
    assert attn.fp8_workspace_bytes(1, 1, 16, 128) == 128 * 16
    for bad in [(1, 1, 16, 64), (1, 1, 16, 96), (-1, 1, 16, 128)]:
        assert attn.fp8_workspace_bytes(*bad) == 0


@pytest.mark.parametrize("args,code", [
    # q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, qd, kd, vd, ws, ws_bytes
    ((0, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, W, 1 << 20), attn.ATTN_EINVAL),   # null q
    ((A, A, A, 2 * A, None, 1, 1, 8, 0, 128, 0.1, 0, 1.0, 1.0, 1.0, W, 1 << 20), attn.ATTN_EINVAL),   # Nk = 0
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 0.0, 1.0, 1.0, W, 1 << 20), attn.ATTN_EINVAL),   # q_descale 0
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, float("inf"), 1.0, W, 1 << 20), attn.ATTN_EINVAL),
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, -2.0, W, 1 << 20), attn.ATTN_EINVAL),  # v_descale < 0
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, 1.0, 1.0, 1.0, W, 1 << 20), attn.ATTN_EUNSUPPORTED),  # D
    ((A + 8, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, W, 1 << 20), attn.ATTN_EUNSUPPORTED),
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, 0, 1 << 20), attn.ATTN_EINVAL),   # no workspace
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, W, 100), attn.ATTN_EINVAL),      # too small
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, W + 4, 1 << 20), attn.ATTN_EUNSUPPORTED),
    ((A, A, A, 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, A, 1 << 20), attn.ATTN_EUNSUPPORTED),  # ws on q
    ((A, A, A, A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, W, 1 << 20), attn.ATTN_EUNSUPPORTED),  # o on q
    ((A, A, A, 2 * A, None, 0, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0, 0, 0), attn.ATTN_OK),             # empty
])
def test_fp8_validation_without_device(lib, args, code):
    assert attn.attn_fwd_fp8(*args, None) == code


def test_fp8_binding_refuses_fp16(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 4, 128, dtype=torch.float16)
    with pytest.raises(TypeError):
        attn.fwd_fp8(x, x, x)


def test_debug_pack_validation(lib):
    assert lib.attn_debug_pack_e4m3(None, None, 4, None) == attn.ATTN_EINVAL
    assert lib.attn_debug_pack_e4m3(A, A, -1, None) == attn.ATTN_EINVAL
    assert lib.attn_debug_pack_e4m3(A, A, 0, None) == attn.ATTN_OK


@pytest.mark.parametrize("args,code", [
    # qh, kh, vh, oh, lh, qd, kd, vd, od, ld, B, H, Nq, Nk, D, scale, causal, chunks
    ((0, W, W, W, None, A, A + (1 << 16), A + (2 << 16), 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, 0), attn.ATTN_EINVAL),
    ((W, W, W, W, W, A, A + (1 << 16), A + (2 << 16), 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, 0), attn.ATTN_EINVAL),
    ((W, W, W, W, None, A, A + (1 << 16), A + (2 << 16), 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, 65), attn.ATTN_EINVAL),
    ((W, W, W, W, None, A, A + (1 << 16), A + (2 << 16), 2 * A, None, 1, 1, 8, 8, 96, 0.1, 0, 0), attn.ATTN_EUNSUPPORTED),
    ((W, W, W, W, None, A, A, A + (2 << 16), 2 * A, None, 1, 1, 8, 8, 64, 0.1, 0, 0), attn.ATTN_EUNSUPPORTED),  # q_dev = k_dev
    ((W, W, W, W, None, A, A + (1 << 16), A + (2 << 16), A, None, 1, 1, 8, 8, 64, 0.1, 0, 0), attn.ATTN_EUNSUPPORTED),
    ((W, W, W, W, None, A, A + (1 << 16), A + (2 << 16), 2 * A, None, 0, 1, 8, 8, 64, 0.1, 0, 0), attn.ATTN_OK),
])
def test_host_entry_validation_without_device(lib, args, code):
    assert attn.attn_fwd_host(*args, None) == code


def test_fp8_host_entry_validation_without_device(lib):
    f = attn.attn_fwd_fp8_host
    base = (W, W, W, W, None, A, A + (1 << 16), A + (2 << 16), 2 * A, None, 1, 1, 8, 8, 128, 0.1, 0, 1.0, 1.0, 1.0)
    ws = (1 << 40, 1 << 20)
    assert f(*((0,) + base[1:]), *ws, 0, None) == attn.ATTN_EINVAL                        # null host q
    assert f(*(base[:4] + (W,) + base[5:]), *ws, 0, None) == attn.ATTN_EINVAL             # lse_host without lse_dev
    assert f(*base, *ws, 65, None) == attn.ATTN_EINVAL                                   # too many chunks
    assert f(*(base[:14] + (64,) + base[15:]), *ws, 0, None) == attn.ATTN_EUNSUPPORTED   # D = 64
    assert f(*(base[:17] + (0.0,) + base[18:]), *ws, 0, None) == attn.ATTN_EINVAL        # q_descale 0
    assert f(*(base[:6] + (A,) + base[7:]), *ws, 0, None) == attn.ATTN_EUNSUPPORTED      # k_dev = q_dev
    assert f(*base, 0, 0, 0, None) == attn.ATTN_EINVAL                                   # no workspace


def test_launch_count_argument_checks_without_device(lib):
    assert attn.fwd_launch_count(1, 4, 128, 128, 96, False) == -attn.ATTN_EINVAL
    assert attn.fwd_launch_count(1, 4, 128, 0, 128, False) == -attn.ATTN_EINVAL
    assert attn.fwd_launch_count(0, 4, 128, 128, 128, False) == 0
