"""Parity of the CUDA forward with the fp64 oracle, element by element.

Small shapes and the three smaller workloads (up to [1,16,8192,128]) are
compared in full (spanning many 128-row / 128-key tiles with ragged tails);
the two largest workloads run at their full sizes, in the same launch the
benchmark times, and are compared on sampled rows, each of which the oracle
computes exactly.
"""
import math

import numpy as np
import pytest

import oracle
from attention_forward_12_gb300 import synth
from gpu_common import compare, full_parity, run_gpu, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch_cuda()
    import attention_forward_12_gb300 as attn
    attn.build()
    attn.load_library()


def test_sdpa_l_listing_shape():
    w = synth.WORKLOADS["sdpa_l_1x4x128x64"]
    full_parity(w.B, w.H, w.Nq, w.Nk, w.D, w.causal, w.seed)


def test_sdpa_p_benchmark_shape_full():
    w = synth.WORKLOADS["sdpa_p_1x8x4096x64"]
    full_parity(w.B, w.H, w.Nq, w.Nk, w.D, w.causal, w.seed)


EDGE = [
    # B, H, Nq, Nk, D, causal
    (1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 1, 17, 17, 64, True),
    (1, 2, 128, 128, 128, False),
    (1, 1, 129, 129, 64, True),
    (2, 1, 255, 300, 128, False),
    (1, 1, 300, 255, 128, True),
    (1, 3, 383, 129, 64, True),
    (3, 2, 200, 1000, 64, False),
    (1, 1, 640, 640, 128, True),
    (2, 2, 1000, 1, 128, False),
    (1, 1, 513, 2049, 128, False),
    (1, 1, 2049, 513, 64, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,D,causal", EDGE)
def test_edge_shapes(B, H, Nq, Nk, D, causal):
    full_parity(B, H, Nq, Nk, D, causal, seed=1000 + Nq + 7 * Nk + D)


@pytest.mark.parametrize("B,H,Nq,Nk,D", [
    (1, 80, 300, 2100, 128),  # 160 half-empty pairs: all 240 query tiles as single-tile CTAs
    (1, 3, 1000, 777, 128),   # 12 pairs, all as single query tiles (an odd key tile count per tile)
    (2, 40, 512, 2049, 128),  # 160 pairs, 17 key tiles each: warpgroup 0 holds the ragged one
    (1, 80, 300, 2100, 64),   # the same at D=64 (single-tile CTAs with two score slots)
    (1, 40, 300, 2100, 128),  # 80 half-empty pairs, below a wave: single-tile CTAs
    (1, 3, 1000, 777, 64),
])
def test_partial_last_wave_as_single_query_tiles(B, H, Nq, Nk, D):
    """Non-causal: the pairs of a last wave that would fill at most half the
    SMs are re-run as CTAs of one query tile, both warpgroups sharing its key
    tiles and merging their carriers (every other shape of these tests with
    few heads takes that path too).  After full waves of pairs this needs 16
    key tiles or more per query tile.  Grids of half-empty pairs run as
    single-tile CTAs alone when that takes clearly fewer waves."""
    full_parity(B, H, Nq, Nk, D, False, seed=500 + H + Nk + D)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True)])
def test_peaked_scores_small(D, causal):
    """Q, K ~ N(0, 3^2): sharply peaked rows, the running max jumps often."""
    full_parity(1, 2, 700, 900, D, causal, seed=77, sigma_qk=3.0)


def _sampled(name, n_random=4096):
    w = synth.WORKLOADS[name]
    q, k, v = synth.workload_qkv(w)
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    rows = synth.sample_rows(w.B, w.H, w.Nq, n_random, w.seed, w.causal)
    O, L, _ = oracle.attn_rows(q, k, v, w.scale, w.causal, rows)
    return compare(o.reshape(-1, w.D)[rows], lse.reshape(-1)[rows], O, L, name)


def test_long_1x16x8192x128_full():
    """Every row of the [1,16,8192,128] workload (0.55 TFLOP of fp64 oracle)."""
    w = synth.WORKLOADS["long_1x16x8192x128"]
    full_parity(w.B, w.H, w.Nq, w.Nk, w.D, w.causal, w.seed, w.sigma_qk, w.sigma_v, w.scale)


def test_causal_2x16x16384x128_sampled():
    _sampled("causal_2x16x16384x128")


def test_peaked_4x32x16384x128_sampled():
    _sampled("peaked_4x32x16384x128")


# ------------------------------------------------------------ degenerate cases

def _run_and_compare(q, k, v, scale, causal, label):
    o, lse = run_gpu(q, k, v, scale, causal)
    O, L = oracle.attn_full(q, k, v, scale, causal)
    return compare(o, lse, O, L, label)


def test_all_scores_tied():
    """Every key row identical: all scores of a row tie, O is the mean of V."""
    B, H, N, D = 1, 2, 300, 64
    q = synth.normal_fp16((B, H, N, D), 1.0, 5, 0)
    k = np.broadcast_to(synth.normal_fp16((1, 1, 1, D), 1.0, 5, 1), (B, H, N, D)).copy()
    v = synth.normal_fp16((B, H, N, D), 1.0, 5, 2)
    _run_and_compare(q, k, v, 0.125, False, "tied")
    _run_and_compare(q, k, v, 0.125, True, "tied causal")


def test_scale_zero_uniform():
    q, k, v = synth.make_qkv(1, 1, 257, 333, 128, 9)
    _run_and_compare(q, k, v, 0.0, False, "scale 0")
    _run_and_compare(q, k, v, 0.0, True, "scale 0 causal")


def test_one_dominant_key():
    B, H, N, D = 1, 1, 512, 128
    q = np.full((B, H, N, D), 0.25, np.float16)
    k = synth.normal_fp16((B, H, N, D), 0.1, 6, 1)
    k[0, 0, 333] = 2.0  # score 0.25*2*128*scale: dominates every row
    v = synth.normal_fp16((B, H, N, D), 1.0, 6, 2)
    _run_and_compare(q, k, v, 1.0 / math.sqrt(D), False, "dominant key")


@pytest.mark.parametrize("D", [64, 128])
def test_running_max_grows_every_tile(D):
    """Scores rise along the keys by more than the lazy-rescale threshold per
    tile, so every tile rescales O."""
    B, H, N = 1, 2, 1024
    q = np.full((B, H, N, D), 0.5, np.float16)
    ramp = (np.arange(N, dtype=np.float64) / N * 16.0).astype(np.float16)  # 0 .. 16
    k = np.broadcast_to(ramp[None, None, :, None], (B, H, N, D)).astype(np.float16).copy()
    k += synth.normal_fp16((B, H, N, D), 0.05, 7, 1)
    v = synth.normal_fp16((B, H, N, D), 1.0, 7, 2)
    # score = 0.5 * D * ramp / sqrt(D) = 4 * ramp (D=64) or 5.7 * ramp (D=128):
    # 11.5 or 16 log2 units per 128 keys
    _run_and_compare(q, k, v, 1.0 / math.sqrt(D), False, "growing max")
    _run_and_compare(q, k, v, 1.0 / math.sqrt(D), True, "growing max causal")


@pytest.mark.parametrize("D", [64, 128])
def test_large_magnitudes(D):
    """Q, K ~ N(0, 8^2) and V ~ N(0, 30^2): the O max-abs bound scales with
    the standard deviation of V (compare's sigma_v), the others do not."""
    full_parity(1, 1, 384, 384, D, False, 10, sigma_qk=8.0, sigma_v=30.0)


def test_deterministic_and_lse_optional():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    q, k, v = (torch.from_numpy(x).cuda() for x in synth.make_qkv(2, 2, 333, 444, 128, 11))
    o1, l1 = attn.fwd(q, k, v, causal=True)
    o2, l2 = attn.fwd(q, k, v, causal=True)
    o3, l3 = attn.fwd(q, k, v, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


def test_side_stream():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    qn, kn, vn = synth.make_qkv(1, 2, 600, 700, 64, 12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
        o, lse = attn.fwd(q, k, v, causal=False)
    s.synchronize()
    assert attn.get_status(s.cuda_stream) == attn.ATTN_OK
    O, L = oracle.attn_full(qn, kn, vn, 0.125, False)
    compare(o.cpu().numpy(), lse.cpu().numpy(), O, L, "side stream")


@pytest.mark.parametrize("B,H,Nq,Nk,D", [(2, 40, 512, 2049, 128), (1, 16, 8192, 8192, 64)])
def test_stream_order_after_the_dependent_launch(B, H, Nq, Nk, D):
    """A launch of pairs followed by a dependent single-tile launch: work
    queued after the forward on the same stream, with no synchronisation in
    between, must see all of O (the single-tile CTAs wait for the pairs'
    grid before they exit).  Copies taken at once, several times, must equal
    the output read after a synchronisation."""
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    assert attn.fwd_launch_count(B, H, Nq, Nk, D, False) == 2
    qn, kn, vn = synth.make_qkv(B, H, Nq, Nk, D, seed=77)
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    copies = []
    for _ in range(4):
        o.fill_(float("nan"))
        attn.fwd(q, k, v, causal=False, out=o, lse=lse)
        copies.append((o.clone(), lse.clone()))  # same stream, no synchronisation
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    for oc, lc in copies:
        assert torch.equal(oc, o) and torch.equal(lc, lse)
    assert not torch.isnan(o).any()


def test_argument_errors_on_device():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    q = torch.zeros(1, 1, 64, 64, dtype=torch.float16, device="cuda")
    buf = torch.zeros(64 * 64 + 8, dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    p = q.data_ptr()
    f = attn.attn_fwd
    assert f(p, p, p, o.data_ptr(), None, 1, 1, 64, 64, 64, 0.125, False, None) == attn.ATTN_OK
    assert f(p, p, p, buf.data_ptr() + 2, None, 1, 1, 64, 64, 64, 0.125, False, None) == attn.ATTN_EUNSUPPORTED
    assert f(p, p, p, p, None, 1, 1, 64, 64, 64, 0.125, False, None) == attn.ATTN_EUNSUPPORTED  # o aliases q
    assert f(p, p, p, o.data_ptr(), None, 1, 1, 64, 0, 64, 0.125, False, None) == attn.ATTN_EINVAL
    assert f(p, p, p, o.data_ptr(), None, 1, 1, 64, 64, 96, 0.125, False, None) == attn.ATTN_EUNSUPPORTED
    assert f(p, p, p, o.data_ptr(), None, 0, 1, 64, 64, 64, 0.125, False, None) == attn.ATTN_OK
    assert f(p, p, p, o.data_ptr(), None, 1, 1, 64, 64, 64, -1.0, False, None) == attn.ATTN_EINVAL
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK


# ------------------------------------------------------------ maximum sizes

@pytest.mark.parametrize("causal", [False, True])
def test_max_heads_grid_limit(causal):
    """B*H = 65535, the largest head count the grid takes: every (b, h) is its
    own problem; compared in full (three query rows, three keys each)."""
    B, H, Nq, Nk, D = 3, 21845, 3, 3, 64
    q, k, v = synth.make_qkv(B, H, Nq, Nk, D, seed=41)
    o, lse = run_gpu(q, k, v, 0.125, causal)
    O, L = oracle.attn_full(q, k, v, 0.125, causal)
    compare(o, lse, O, L, f"B*H = 65535, causal={causal}")


@pytest.mark.parametrize("B,H,Nq,Nk,D", [
    (2, 40, 700, 700, 128),   # 80 heads x 3 pairs, the last pair ragged
    (2, 40, 700, 700, 64),
    (1, 80, 1300, 900, 128),  # Nq > Nk: the last query tiles see every key
    (3, 30, 520, 1100, 64),   # Nq < Nk
])
def test_causal_pairs_heaviest_first_across_heads(B, H, Nq, Nk, D):
    """Causal CTAs take the pairs of all heads in decreasing pair order (the
    linear CTA index mapped pair-major): every (head, pair) must be computed
    exactly once, ragged pairs included; compared in full.  (More than half
    a wave of pairs, so these run as pair CTAs.)"""
    full_parity(B, H, Nq, Nk, D, True, seed=700 + B * H + Nq + D)


@pytest.mark.parametrize("B,H,Nq,Nk,D", [
    (1, 2, 1000, 1000, 128),  # 8 pairs: 16 single-tile CTAs, the last tile ragged
    (1, 4, 2048, 2048, 64),
    (2, 3, 700, 900, 128),    # Nq < Nk
    (1, 1, 4096, 4096, 128),  # one head, 32 query tiles of 1..32 key tiles
    (1, 3, 900, 300, 64),     # Nq > Nk
    (1, 8, 4096, 4096, 64),   # 128 pairs: 256 single-tile CTAs, heaviest first over two waves
    (2, 4, 3000, 3000, 128),  # 96 pairs, the last query tile of each head ragged
])
def test_causal_small_grids_as_single_query_tiles(B, H, Nq, Nk, D):
    """Causal grids of at most one wave of pairs run as single-query-tile
    CTAs, heaviest first across heads (the two warpgroups alternate the
    tile's key tiles, the diagonal one masked in whichever takes it, and
    merge their carriers); compared in full."""
    full_parity(B, H, Nq, Nk, D, True, seed=900 + B * H + Nq + Nk + D)


@pytest.mark.parametrize("Nk,D", [(1 << 16, 64), (1 << 18, 64), (1 << 19, 64), (1 << 19, 128)])
def test_long_key_ranges(Nk, D):
    """Up to 2^19 keys -- the most one pass may accumulate per row -- for a few
    query rows: 4096 key tiles in one CTA's loop."""
    B, H, Nq = 1, 1, 3
    scale = 1.0 / math.sqrt(D)
    q, k, v = synth.make_qkv(B, H, Nq, Nk, D, seed=42, sigma_qk=2.0)
    o, lse = run_gpu(q, k, v, scale, False)
    O, L = oracle.attn_full(q, k, v, scale, False)
    compare(o, lse, O, L, f"Nk = {Nk}, D = {D}")


def test_million_keys_are_refused_by_the_single_pass():
    """2^20 keys per row would drift past the relative-RMS bound in one pass:
    attn_fwd refuses it (nothing enqueued) and points to split-KV."""
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    q = torch.zeros(1, 1, 3, 64, dtype=torch.float16, device="cuda")
    kv = torch.zeros(1, 1, 1 << 20, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.fwd(q, kv, kv, scale=0.125)
    assert e.value.code == attn.ATTN_ETOOLONG
    # causal: the rows accumulate min(Nk, i + 1) keys, so a short query block passes
    o, _ = attn.fwd(q, kv, kv, scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    with pytest.raises(attn.AttnError) as e:  # one share of 2^20 keys is a single pass too
        attn.fwd_splitkv(q, kv, kv, scale=0.125, num_splits=1)
    assert e.value.code == attn.ATTN_ETOOLONG


def test_million_keys_through_split_kv():
    """2^20 keys: beyond ~2^19 keys the single pass's fp32 tensor-core
    accumulation of O drifts past the relative-RMS bound, so key ranges this
    long go through split-KV (16 shares of 2^16 keys, merged in fp32)."""
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    B, H, Nq, Nk, D = 1, 1, 3, 1 << 20, 64
    qn, kn, vn = synth.make_qkv(B, H, Nq, Nk, D, seed=42, sigma_qk=2.0)
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, kn, vn))
    o, lse = attn.fwd_splitkv(q, k, v, scale=0.125, num_splits=16)
    torch.cuda.synchronize()
    assert attn.get_status() == attn.ATTN_OK
    O, L = oracle.attn_full(qn, kn, vn, 0.125, False)
    compare(o.cpu().numpy(), lse.cpu().numpy(), O, L, "Nk = 2^20, split-KV x16")


def test_over_65535_is_rejected_before_launch():
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    q = torch.zeros(1, 65536, 1, 64, dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    rc = attn.attn_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None, 1, 65536, 1, 1, 64,
                       0.125, False, None)
    assert rc == attn.ATTN_EUNSUPPORTED


@pytest.mark.parametrize("causal", [False, True])
def test_huge_jump_of_the_running_max(causal):
    """Scores jump by ~130 log2 units after the first 200 keys: exponentials
    taken against the old reference would overflow, so the row update must
    redo the tile against the new one."""
    B, H, N, D = 1, 2, 640, 128
    q = np.full((B, H, N, D), 1.0, np.float16)
    k = synth.normal_fp16((B, H, N, D), 0.05, 8, 1)
    k[:, :, 200:] += np.float16(8.0)
    v = synth.normal_fp16((B, H, N, D), 1.0, 8, 2)
    _run_and_compare(q, k, v, 1.0 / math.sqrt(D), causal, "huge jump")


def test_launch_count_reports_the_single_tile_launch():
    """attn_fwd_launch_count: two kernels exactly when the non-causal
    forward re-runs a last partial wave of at most half the SMs as
    single-query-tile CTAs next to full waves of pairs; one otherwise
    (causal grids below half a wave are one launch of single-tile CTAs)."""
    torch = torch_cuda()
    import attention_forward_12_gb300 as attn
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def expected(B, H, Nq, Nk, D, causal):
        pairs = B * H * ((Nq + 255) // 256)
        if causal:  # pairs, or single-tile CTAs alone up to one wave: one launch either way
            return 1
        last = pairs % sms
        tail = last if (last > 0 and 2 * last <= sms) else 0
        if 0 < tail < pairs and (Nk + 127) // 128 < 16:  # short CTAs: no second launch after full waves
            tail = 0
        # all single-tile CTAs when the existing query tiles take clearly fewer waves that way
        q_tiles = B * H * ((Nq + 127) // 128)
        waves_now = -(-(pairs - tail) // sms) + (0.65 if tail else 0.0)
        if 0.65 * -(-q_tiles // sms) < 0.9 * waves_now:
            tail = pairs
        return int(pairs - tail > 0) + int(tail > 0)

    for (B, H, Nq, Nk, D, causal) in [(1, 16, 8192, 8192, 128, False), (4, 32, 16384, 16384, 128, False),
                                      (1, 4, 512, 8192, 128, False), (2, 16, 16384, 16384, 128, True),
                                      (1, 8, 4096, 4096, 64, False), (1, 80, 300, 300, 128, False),
                                      (1, 80, 300, 4096, 128, False), (2, 40, 512, 512, 64, False),
                                      (1, 2, 1000, 1000, 128, True), (1, 40, 300, 2100, 128, False),
                                      (2, 40, 512, 2049, 128, False)]:
        assert attn.fwd_launch_count(B, H, Nq, Nk, D, causal) == expected(B, H, Nq, Nk, D, causal)
    assert attn.fwd_launch_count(0, 4, 128, 128, 128, False) == 0
    assert attn.fwd_launch_count(1, 4, 128, 128, 96, False) == -attn.ATTN_EINVAL
