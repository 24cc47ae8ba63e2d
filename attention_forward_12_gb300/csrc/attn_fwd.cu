// attn_fwd.cu -- fused scaled-dot-product attention forward for GB300
// (sm_103a) and its C ABI (include/attn.h).
//
//   O = softmax(scale * Q K^T) V,   LSE = log sum_j exp(scale * q.k_j)
//
// The method is the streaming reduction of "Learning FlashAttention the
// Hard Way -- Part 2": each query row carries (m, d, o) -- running maximum,
// running denominator, running unnormalised output -- across key/value
// tiles, so the N x N scores never reach HBM (sections "Move 0" FA-1 and
// "Move 1 -- Tensor Cores").  The page's kernels are mma.sync designs for
// sm_120; this one is built for the datacenter Blackwell tensor core.
//
// One CTA owns two 128-row query tiles of one (batch, head) -- the
// register-tiling idea of the page's "Move 4" (two independent (m, l, O)
// chains sharing every K/V fragment), lifted to two warpgroups sharing every
// K/V shared-memory tile:
//
//   * TMA producer (warp 8): loads both Q tiles once and streams K and V
//     tiles through an NS-deep ring of 128B-swizzled shared-memory stages,
//     each stage guarded by full/empty mbarriers ("New Hardware: TMA": box
//     copies, hardware swizzle, one issuing thread, mbarrier transaction
//     counts; "Move 3 -- Pipelining": prefetch under compute).
//   * MMA issuer (warp 9; lane 0 issues): S_w = Q_w K_j^T with tcgen05.mma
//     (A and B from shared memory) into TMEM buffer w, and O_w += P_w V_j
//     with tcgen05.mma taking P_w from TMEM, where the softmax wrote it over
//     S_w (the analogue of the page's C->A register repack: P never goes
//     through shared memory).  Issue order per key tile j:
//         O_0 += P_0 V_j,  S_0 = Q_0 K_{j+1}^T,  O_1 += P_1 V_j,  S_1 = Q_1 K_{j+1}^T
//     so that one warpgroup's softmax runs while the tensor core works on
//     the other's tile.  With SPLIT_P (the fp16 D = 128 kernels) each
//     O_w += P_w V_j is issued in two halves of 64 keys: the first as soon
//     as the softmax has released the first half of P_w, overlapping the
//     second half's exponentials -- this shortens each warpgroup's chain
//     softmax -> P V -> Q K^T, which bounds the kernel.  At D = 64 the
//     rotating score slots (below) already take S off that chain, and P is
//     released whole: the second release and its wait cost more there than
//     the overlap returns.
//   * Softmax warpgroups w = 0, 1 (warps 4w..4w+3; thread t owns row t of
//     query tile w, which is TMEM lane t): tcgen05.ld.red of S_w, which
//     returns the row maximum with the scores (masked tiles: mask, then a
//     3-input max pass), p = 2^(s*scale*log2(e) - m) with the scale
//     folded into a packed FFMA2, packed row sums, fp16 pack of p written
//     back over S_w (in two released halves with SPLIT_P, the O rescale
//     running between them; otherwise after the exponentials).  O_w is
//     rescaled lazily, before the tile's P is released: only when a row's
//     maximum grows by more than kTau (log2 units) over the reference it
//     was using;
//     otherwise p is taken against the stale reference, which is exact
//     because p, d and o share it (the conditional rescale the page credits
//     to FlashAttention-4 in "Relationship to FA-3 and FA-4").  At the end the
//     warpgroup normalises O_w by d and writes fp16 O (staged in its query
//     tile's shared-memory buffer and stored with TMA) and fp32 LSE.
//   * Causal (key j masked when j > i): each query tile visits only the key
//     tiles up to its own diagonal; only the diagonal and the ragged last
//     tile take the masked path.
//
//   * Wave quantisation (single pass, fp16 and E4M3): when a launch's last
//     wave of CTAs would occupy at most half the SMs, its pairs run as a
//     second launch of CTAs that each take one query tile, the two
//     warpgroups alternating its key tiles and merging their carriers at
//     the end -- twice the CTAs, half the work each.  Causal: only grids
//     of at most one wave of pairs, which run as single-tile CTAs alone.
//
// TMEM (512 columns): at D = 128, S_0/P_0 [0,128), S_1/P_1 [128,256),
// O_0 [256,384), O_1 [384,512).  At D = 64 three score slots [0,128),
// [128,256), [256,384) rotate between the two query tiles (so a tile's next
// scores do not wait for its own P V), O_0 [384,448), O_1 [448,512).
//
// Every mbarrier wait is bounded (see WaitCtl): a wait that runs out raises
// the CTA's abort flag and the device status word; the CTA then drains its
// TMA copies and tensor-core work in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "sm103_primitives.cuh"

using namespace attn_sm103;

namespace {

constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kBlockM = 128;           // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;           // keys per tile
constexpr int kRowsPerCta = 2 * kBlockM;
constexpr float kTau = 8.0f;           // lazy-rescale threshold, log2 units
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 64 fp16 (one swizzle column block)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// Exponentials sent to the FMA-pipe polynomial: one pair in kEmu (0 = none).
constexpr int kEmu64 = 0;
constexpr int kEmu128 = 0;
// The share attn_debug_fwd_poly_exp sends there (one pair in four), so that
// the polynomial's device code runs inside the forward under test.
constexpr int kDebugEmu = 4;

template <int HD, int NS, bool FP8 = false, int QT = 2>
struct Layout {
  static constexpr int kElem = FP8 ? 1 : 2;                   // bytes per element
  static constexpr int kChunks = HD * kElem / 128;            // 128-byte column blocks per row
  static constexpr int kChunkElems = 128 / kElem;
  static constexpr uint32_t kTileBytes = kBlockM * HD * kElem;  // one Q, K or V tile
  // QT query tiles, then NS K and NS V stages; q_full, k/v full/empty[NS],
  // s_full/p_half/p_full[3] (one per TMEM score slot), o_done[4], drain,
  // xchg, o_staged[2]; then the TMEM address, the abort flag and the last
  // loads per stage
  static constexpr int kBars = 1 + 4 * NS + 3 * 3 + 4 + 1 + 1 + 2;
  static constexpr size_t kSmem = 1024 + kTileBytes * (QT + 2 * NS) + kBars * 8 + 8 + 8 + NS * 8;
};

// K/V ring depth of the single-tile CTAs.  They hold one query tile, so at
// fp16 D = 128 the ring takes the second tile's space and grows from 2 to 3
// stages of 64 KB: a V stage is then free a tile earlier, and the loads of
// the tile after next no longer wait for the last product.  The 16 KB-tile
// kernels (D = 64, E4M3) keep the pairs' 4 stages: 6 measured no faster.
template <int HD, bool FP8>
constexpr int single_stages() { return (HD == 128 && !FP8) ? 3 : 4; }

// Key tiles query tile w of the CTA visits (0 if the tile lies past Nq).
template <bool CAUSAL>
__device__ __forceinline__ int tile_kv_count(int row0, int Nq, int Nk) {
  if (row0 >= Nq) return 0;
  const int kv_end = CAUSAL ? min(Nk, row0 + kBlockM) : Nk;
  return (kv_end + kBlockN - 1) / kBlockN;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// p = 2^(s*sl2 - m_ref) for one 128-column score row (sr, TMEM columns
// tS .. tS + 127), packed to fp16 pairs (FP8: E4M3 quadruples) and written
// back over S in two halves of 64 keys; with SPLIT_P each half is released
// to the MMA thread as soon as it is in TMEM, `mid` running just before the
// first release.  Returns the row sum of the fp32 p.  MASK: 0 = columns
// >= lim masked when `masked` (decided at run time), 1 = none masked, 2 =
// columns >= lim masked.  EARLY (fp16): each 32 keys of P go to TMEM as soon
// as they are packed, instead of one store per half.
template <int MASK, int EMU, int SPLIT_P, bool FP8, bool EARLY, typename Mid>
__device__ __forceinline__ float exp_row(const uint32_t (&sr)[4][32], float2 sl2v, float2 nm, bool masked, int lim,
                                         uint32_t tS, uint64_t* p_half, uint64_t* p_full, Mid&& mid) {
  const bool mk = MASK == 2 || (MASK == 0 && masked);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[FP8 ? 16 : 32];
    uint32_t pq[2][16];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * h + cc;
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float p[4];
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
          const float2 x =
              __ffma2_rn(make_float2(__uint_as_float(sr[c][e + q]), __uint_as_float(sr[c][e + q + 1])), sl2v, nm);
          if (EMU > 0 && ((e + q) >> 1) % (EMU > 0 ? EMU : 1) == (EMU > 0 ? EMU : 1) - 1) {
            const float2 pp = exp2_poly2(x);  // one pair in EMU on the FMA pipe
            p[q] = pp.x;
            p[q + 1] = pp.y;
          } else {
            p[q] = ex2_approx(x.x);
            p[q + 1] = ex2_approx(x.y);
          }
          if (MASK != 1 && mk) {  // -inf * 0 is NaN when scale == 0: select explicitly
            p[q] = (c * 32 + e + q < lim) ? p[q] : 0.f;
            p[q + 1] = (c * 32 + e + q + 1 < lim) ? p[q + 1] : 0.f;
          }
          acc[((e + q) >> 1) & 3] = __fadd2_rn(acc[((e + q) >> 1) & 3], make_float2(p[q], p[q + 1]));
        }
        if constexpr (FP8) {
          pk[cc * 8 + (e >> 2)] = pack_e4m3x4(p[0], p[1], p[2], p[3]);
        } else if constexpr (EARLY) {
          pq[cc][e >> 1] = pack_half2(p[0], p[1]);
          pq[cc][(e >> 1) + 1] = pack_half2(p[2], p[3]);
        } else {
          pk[cc * 16 + (e >> 1)] = pack_half2(p[0], p[1]);
          pk[cc * 16 + (e >> 1) + 1] = pack_half2(p[2], p[3]);
        }
      }
      if constexpr (!FP8 && EARLY) tmem_st16(tS + h * 32 + cc * 16, pq[cc]);
    }
    if constexpr (FP8) {
      tmem_st16(tS + h * 16, pk);
    } else if constexpr (!EARLY) {
      tmem_st32(tS + h * 32, pk);
    }
    if constexpr (SPLIT_P) {
      if (h == 0) mid();  // runs before the first half is released
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(h ? p_full : p_half);
    }
  }
  const float2 a01 = __fadd2_rn(acc[0], acc[1]);
  const float2 a23 = __fadd2_rn(acc[2], acc[3]);
  const float2 a = __fadd2_rn(a01, a23);
  return a.x + a.y;
}

}  // namespace

// Device status word: 0 = ok, otherwise the first ATTN_E* code a kernel
// recorded since the last attn_get_status().
__device__ int g_attn_status;

template <int HD, bool CAUSAL, int NS, int SPLIT_P, int EMU, bool SPLITKV, bool FP8, int SLOTS, bool SINGLE>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                __half* __restrict__ out,
                float* __restrict__ lse, float* __restrict__ ws_o, float* __restrict__ ws_l, int Nq, int Nk,
                float sl2, float o_scale, int* status_host, uint64_t timeout_ns,
                int drop_tile, int n_main) {
  static_assert(!FP8 || HD == 128, "the E4M3 kernel is built for D = 128 only");
  static_assert(SPLIT_P == 0 || SPLIT_P == 2, "P released whole (0) or in two halves (2)");
  constexpr int QT = SINGLE ? 1 : 2;  // query tiles held in shared memory
  using L = Layout<HD, NS, FP8, QT>;
  constexpr uint32_t TB = L::kTileBytes;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sQ = sm;                 // QT tiles
  uint8_t* sK = sQ + QT * TB;       // NS tiles
  uint8_t* sV = sK + NS * TB;       // NS tiles
  uint64_t* q_full = reinterpret_cast<uint64_t*>(sV + NS * TB);
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;  // [SLOTS] S landed in TMEM score slot b
  uint64_t* p_half = s_full + 3;    // [SLOTS] first 64 keys of P written over slot b (and O rescaled)
  uint64_t* p_full = p_half + 3;    // [SLOTS] all of P written over slot b
  uint64_t* o_done = p_full + 3;    // [4] completed O_w += P_w V_j: SLOTS = 2: [w], one phase per
                                    // product; SLOTS = 3: [2w + (j & 1)], one phase per two
  uint64_t* drain = o_done + 4;     // abort path only
  uint64_t* xchg = drain + 1;       // single-tile CTA: both warpgroups' (m, d) written
  uint64_t* o_staged = xchg + 1;    // [2] fp16 O tile w staged in shared memory for its TMA store
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_staged + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* last_k = abort_flag + 1;     // [NS] last tile loaded per stage (abort drain)
  int* last_v = last_k + NS;
  // Single-tile CTA: the (m, d) exchange of the two warpgroups, in the
  // query tile's buffer, which is free once every product has completed.
  float* x_m = reinterpret_cast<float*>(sQ);  // [2][128] m per warpgroup and row
  float* x_d = x_m + 2 * kBlockM;             // [2][128] d per warpgroup and row

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work of this CTA.  Usually two query tiles of one (batch, head) -- a
  // pair -- each warpgroup taking one of them against every key tile (of the
  // share, with split-KV).  SINGLE (the single pass):
  // one query tile, both warpgroups sharing its key range -- warpgroup w
  // takes key tiles w, w + 2, ... -- and merging their two partial results
  // at the end.  The host runs the pairs of a last partial wave that would
  // occupy at most half the SMs this way, as a second launch of twice as
  // many CTAs doing half the work each: the pairs' launch skips them
  // (n_main: the pairs it keeps, in (head, pair) order), and the single-
  // tile launch's CTA b takes query tile b % 2 of pair n_main + b / 2.
  // Small grids, grids of half-empty pairs and causal grids of at most one
  // wave of pairs run as single-tile CTAs alone (n_main = 0).
  constexpr bool single = SINGLE;
  static_assert(!SINGLE || (SLOTS == 2 && !SPLITKV), "single-tile CTAs");
  int bh, pair, half = 0;
  if constexpr (SINGLE) {
    const int n_pairs = (Nq + kRowsPerCta - 1) / kRowsPerCta;
    const int b = static_cast<int>(blockIdx.x);
    if constexpr (CAUSAL) {
      // The whole grid (n_main = 0), heaviest query tile first across all
      // heads, as for the causal pairs: a query tile t visits t + 1 key tiles.
      const int nbh = static_cast<int>(gridDim.x) / (2 * n_pairs);
      const int qt = 2 * n_pairs - 1 - b / nbh;
      bh = b % nbh;
      pair = qt >> 1;
      half = qt & 1;
    } else {
      const int item = n_main + (b >> 1);
      half = b & 1;
      pair = item % n_pairs;
      bh = item / n_pairs;
    }
  } else {
    const int lin = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);  // the order CTAs are dispatched in
    if constexpr (CAUSAL) {
      // Causal pairs cost in proportion to their index (pair p visits 2p + 2
      // key tiles).  Heaviest first across all heads: the first CTAs take
      // every head's last pair, then every head's pair before it, and so
      // on, so the light pairs fill the end of the grid (a longest-first
      // list schedule on the SMs as they free up).
      const int nbh = static_cast<int>(gridDim.y);
      pair = static_cast<int>(gridDim.x) - 1 - lin / nbh;
      bh = lin % nbh;
    } else {
      bh = static_cast<int>(blockIdx.y);
      pair = static_cast<int>(blockIdx.x);
      if (lin >= n_main) return;  // left to the single-tile launch
    }
    // A single-tile launch that follows may start once every CTA here has
    // started (no-op without one).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  const int r0 = pair * kRowsPerCta;
  // Key tiles of this CTA: all of the pair's (grid z = 1), or with split-KV
  // the contiguous share [t0, t1) of split blockIdx.z.  nkv0 / nkv1 count the
  // tiles each warpgroup visits in that share (0 if its query tile lies past
  // Nq or, when causal, if its diagonal comes before the share); nkv counts
  // the K/V tiles the producer loads.
  const int nkv0_all = single ? 0 : tile_kv_count<CAUSAL>(r0, Nq, Nk);
  const int nkv1_all = single ? 0 : tile_kv_count<CAUSAL>(r0 + kBlockM, Nq, Nk);
  const int nkv_all = max(nkv0_all, nkv1_all);
  const int t0 = SPLITKV ? static_cast<int>(static_cast<int64_t>(nkv_all) * blockIdx.z / gridDim.z) : 0;
  const int t1 = SPLITKV ? static_cast<int>(static_cast<int64_t>(nkv_all) * (blockIdx.z + 1) / gridDim.z) : nkv_all;
  const int nkv_single = single ? tile_kv_count<CAUSAL>(r0 + half * kBlockM, Nq, Nk) : 0;
  const int nkv0 = single ? (nkv_single + 1) / 2 : SPLITKV ? max(0, min(t1, nkv0_all) - t0) : nkv0_all;
  const int nkv1 = single ? nkv_single / 2 : SPLITKV ? max(0, min(t1, nkv1_all) - t0) : nkv1_all;
  const int nkv = single ? nkv_single : max(nkv0, nkv1);
  const size_t rows_total = static_cast<size_t>(gridDim.y) * Nq;  // split-KV part stride

  // A CTA of a launch that already recorded an error does no work: after a
  // timeout the remaining CTAs exit at once instead of each waiting out its
  // own limit.  The status word is read by one thread and broadcast.
  if (threadIdx.x == 0) *abort_flag = *static_cast<volatile int*>(&g_attn_status);
  __syncthreads();
  if (*abort_flag) return;
  if (single && nkv == 0) return;  // a single query tile past Nq: nothing to do
  if constexpr (SPLITKV) {
    if (nkv == 0) {
      // No admissible key in this share for either tile: an empty part
      // (O = 0, LSE = -inf), which the merge gives zero weight.
      const int i = r0 + static_cast<int>(threadIdx.x);
      if (threadIdx.x < kRowsPerCta && i < Nq) {
        const size_t rr = static_cast<size_t>(blockIdx.z) * rows_total + static_cast<size_t>(bh) * Nq + i;
        float4* dst = reinterpret_cast<float4*>(ws_o + rr * HD);
#pragma unroll 4
        for (int e = 0; e < HD / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        ws_l[rr] = -INFINITY;
      }
      return;
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      last_k[s] = -1;
      last_v[s] = -1;
    }
    for (int b = 0; b < SLOTS; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_half[b], kBlockM);
      mbar_init(&p_full[b], kBlockM);
    }
    for (int b = 0; b < 4; ++b) mbar_init(&o_done[b], 1);
    mbar_init(drain, 1);
    mbar_init(xchg, 2 * kBlockM);
    mbar_init(&o_staged[0], kBlockM);
    mbar_init(&o_staged[1], kBlockM);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = *tmem_slot;
  // TMEM score slots: one per query tile (SLOTS = 2: S_w at column 128 w),
  // or three that the two query tiles' score tiles rotate through (SLOTS =
  // 3, D = 64: slots at 0, 128, 256).  O_w after the slots.
  constexpr uint32_t kOCol = SLOTS == 3 ? 384 : 256;
  constexpr uint32_t kOStride = SLOTS == 3 ? HD : 128;
  static_assert(SLOTS == 2 || (SLOTS == 3 && kOCol + 2 * HD <= kTmemCols), "TMEM budget");
  // With three slots the score tiles are numbered in the order the tensor
  // core computes them -- (tile 0, Q tile 0), (0, 1), (1, 0), (1, 1), ...,
  // then the longer query tile's remaining ones -- and item n uses slot
  // n % 3.  Item n + 3 reuses the slot once O += P V of item n is issued:
  // a query tile's next scores wait for the other tile's product, not for
  // its own.
  const int mmin = min(nkv0, nkv1);
  const int wlong = nkv0 > nkv1 ? 0 : 1;
  const int nitems = nkv0 + nkv1;
  const WaitCtl wc{abort_flag, &g_attn_status, status_host, timeout_ns};

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      // A single-tile CTA loads its one query tile into the first Q buffer,
      // which both warpgroups' Q K^T read.
      const int q0_row = single ? r0 + half * kBlockM : r0;
      const bool load_q1 = !single && nkv1 > 0;
      mbar_arrive_expect_tx(q_full, (nkv0 > 0 ? TB : 0) + (load_q1 ? TB : 0));
      if (nkv0 > 0)
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sQ + c * kChunkBytes, &tmQ, q_full, c * L::kChunkElems, q0_row, bh);
      if (load_q1)
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sQ + TB + c * kChunkBytes, &tmQ, q_full, c * L::kChunkElems, r0 + kBlockM, bh);
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (j >= NS) ok = mbar_wait(&k_empty[s], ph ^ 1, wc, ATTN_ETIMEOUT);
        if (!ok) break;
        if (j != drop_tile) {  // drop_tile >= 0 only under attn_debug_set
          mbar_arrive_expect_tx(&k_full[s], TB);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sK + s * TB + c * kChunkBytes, &tmK, &k_full[s], c * L::kChunkElems, (t0 + j) * kBlockN, bh);
          last_k[s] = j;
        }
        if (j >= NS) ok = mbar_wait(&v_empty[s], ph ^ 1, wc, ATTN_ETIMEOUT);
        if (!ok) break;
        mbar_arrive_expect_tx(&v_full[s], TB);
        if constexpr (FP8) {
          // V^T tile: 128 rows of D, each 128 keys (bytes) long.
          tma_load_3d(sV + s * TB, &tmV, &v_full[s], (t0 + j) * kBlockN, 0, bh);
        } else {
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sV + s * TB + c * kChunkBytes, &tmV, &v_full[s], c * 64, (t0 + j) * kBlockN, bh);
        }
        last_v[s] = j;
      }
      // Tail: wait until the tensor core has released every stage, so that
      // no completion arrives on a barrier after the CTA has exited.
      for (int s = 0; s < NS && ok; ++s) {
        if (last_k[s] >= 0) ok = mbar_wait(&k_empty[s], (last_k[s] / NS) & 1, wc, ATTN_ETIMEOUT);
        if (ok && last_v[s] >= 0) ok = mbar_wait(&v_empty[s], (last_v[s] / NS) & 1, wc, ATTN_ETIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, so that every address and
    // descriptor in it is warp-uniform; lane 0 alone issues (the *_warp
    // forms).  Descriptors are built once and stepped by adding byte
    // offsets / 16 to their start-address field (no carry: shared-memory
    // addresses / 16 fit in its 14 bits).  The base address goes through an
    // opaque move so that the descriptors are built here, not hoisted above
    // the role branch where they would hold registers in the softmax warps.
    uint32_t base;
    asm volatile("mov.u32 %0, %1;" : "=r"(base) : "r"(smem_u32(sQ)));
    constexpr uint32_t kIdescQK = idesc_f16_f32(kBlockM, kBlockN, false, false);
    // fp16: V is MN-major (LBO = next 64 columns of D); E4M3: V^T is
    // K-major like K.  (With format code 0, the E4M3 descriptor bits are
    // those of fp16.)
    constexpr uint32_t kIdescPV = idesc_f16_f32(kBlockM, HD, false, !FP8);
    const uint64_t dQ = smem_desc(base, 16, 1024);
    const uint64_t dK = smem_desc(base + QT * TB, 16, 1024);
    const uint64_t dV = smem_desc(base + (QT + NS) * TB, FP8 ? 16u : kChunkBytes, 1024);
    constexpr int kQkSteps = HD * L::kElem / 32;       // 32 bytes of D per product
    constexpr int kPvSteps = kBlockN * L::kElem / 32;  // 32 bytes of keys per product
    // S_w = Q_w K^T of stage s: both operands K-major, 128B swizzle; the
    // reduction over D runs in steps of 16 (32 bytes inside a swizzle row).
    auto issue_s = [&](int w, int s, int slot) {
      const uint32_t dS = tmem + slot * 128;
      const uint64_t a = dQ + (((single ? 0 : w) * TB) >> 4);  // a single-tile CTA has one Q tile
      const uint64_t b = dK + ((s * TB) >> 4);
#pragma unroll
      for (int kk = 0; kk < kQkSteps; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        if constexpr (FP8)
          umma_ss_f8_warp(dS, a + off, b + off, kIdescQK, kk > 0 ? 1u : 0u);
        else
          umma_ss_warp(dS, a + off, b + off, kIdescQK, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&s_full[slot]);
    };
    // O_w += P_w V of stage s: P (fp16, two per column) from TMEM as the A
    // operand; V MN-major in shared memory (rows = keys, 128 bytes of D per
    // row; LBO = next 64 columns of D, SBO = next 8 keys).  The first 64 keys
    // go as soon as the softmax has released the first half of P, so the
    // tensor core works while the second half is being computed.
    auto issue_pv = [&](int w, int j, int s, int slot, uint32_t par) -> bool {
      const uint32_t aP = tmem + slot * 128;
      const uint32_t dO = tmem + kOCol + w * kOStride;
      const uint64_t b = dV + ((s * TB) >> 4);
      constexpr int kParts = SPLIT_P ? 2 : 1;
#pragma unroll
      for (int part = 0; part < kParts; ++part) {
        const bool last = part == kParts - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(last ? &p_full[slot] : &p_half[slot], par, wc, ATTN_ETIMEOUT)))
          return false;
        tc_fence_after();
#pragma unroll
        for (int kk = part * kPvSteps / kParts; kk < (part + 1) * kPvSteps / kParts; ++kk) {
          // P: 8 TMEM columns (32 bytes of keys) per product.  V: the next
          // 16 keys (fp16, 16 rows of 128 B) or 32 keys (V^T, 32 bytes in).
          if constexpr (FP8)
            umma_ts_f8_warp(dO, aP + kk * 8, b + ((kk * 32) >> 4), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          else
            umma_ts_warp(dO, aP + kk * 8, b + ((kk * 2048) >> 4), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
      }
      umma_commit_warp(&o_done[SLOTS == 3 ? 2 * w + (j & 1) : w]);
      return true;
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar, parity, wc, ATTN_ETIMEOUT))) return false;
      tc_fence_after();
      return true;
    };
    if constexpr (SINGLE) {
      // Single query tile: warpgroup w takes key tiles w, w + 2, ...; key
      // tile t lives in stage t % NS.  Its local tile index jj = t / 2
      // selects the parity of its slot, P and o_done phases (one per tile
      // of that warpgroup).  K stages are released after their Q K^T, V
      // stages after their P V, so the producer's K loads stay a tile pair
      // ahead.
      auto st = [](int t) { return t % NS; };
      auto ph = [](int t) { return static_cast<uint32_t>((t / NS) & 1); };
      bool ok = wait_all(q_full, 0);
      for (int t = 0; t < 2 && t < nkv && ok; ++t) {
        if (!(ok = wait_all(&k_full[st(t)], ph(t)))) break;
        issue_s(t, st(t), t);
        umma_commit_warp(&k_empty[st(t)]);
      }
      for (int t = 0; t < nkv && ok; ++t) {
        const int w = t & 1, jj = t >> 1;
        if (!(ok = wait_all(&v_full[st(t)], ph(t)))) break;
        if (!(ok = issue_pv(w, jj, st(t), w, static_cast<uint32_t>(jj & 1)))) break;
        umma_commit_warp(&v_empty[st(t)]);
        if (t + 2 < nkv) {
          if (!(ok = wait_all(&k_full[st(t + 2)], ph(t + 2)))) break;
          issue_s(w, st(t + 2), w);
          umma_commit_warp(&k_empty[st(t + 2)]);
        }
      }
    } else if constexpr (SLOTS == 2) {
      bool ok = wait_all(q_full, 0) && wait_all(&k_full[0], 0);
      if (ok) {
        if (nkv0 > 0) issue_s(0, 0, 0);
        if (nkv1 > 0) issue_s(1, 0, 1);
        umma_commit_warp(&k_empty[0]);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int s = j % NS;
        const int s1 = (j + 1) % NS;
        const bool more = j + 1 < nkv;
        if (!(ok = wait_all(&v_full[s], (j / NS) & 1))) break;
        if (j < nkv0 && !(ok = issue_pv(0, j, s, 0, j & 1))) break;
        if (more) {
          if (!(ok = wait_all(&k_full[s1], ((j + 1) / NS) & 1))) break;
          if (j + 1 < nkv0) issue_s(0, s1, 0);
        }
        if (j < nkv1 && !(ok = issue_pv(1, j, s, 1, j & 1))) break;
        umma_commit_warp(&v_empty[s]);
        if (more) {
          if (j + 1 < nkv1) issue_s(1, s1, 1);
          umma_commit_warp(&k_empty[s1]);
        }
      }
    } else {
      // Items in order: S of item n + 3 follows O += P V of item n.  A key
      // tile's K stage is released after its last score item, its V stage
      // after its last product.
      auto tile_of = [&](int n, int& j, int& w) {
        if (n < 2 * mmin) {
          j = n >> 1;
          w = n & 1;
        } else {
          j = mmin + (n - 2 * mmin);
          w = wlong;
        }
      };
      auto last_item = [&](int j) { return j < mmin ? 2 * j + 1 : 2 * mmin + (j - mmin); };
      int k_seen = -1, v_seen = -1;  // last key tile whose K / V landing was waited for
      auto s_item = [&](int n) -> bool {
        int j, w;
        tile_of(n, j, w);
        if (j > k_seen) {
          if (!wait_all(&k_full[j % NS], (j / NS) & 1)) return false;
          k_seen = j;
        }
        issue_s(w, j % NS, n % 3);
        if (n == last_item(j)) umma_commit_warp(&k_empty[j % NS]);
        return true;
      };
      bool ok = wait_all(q_full, 0);
      for (int n = 0; n < 3 && n < nitems && ok; ++n) ok = s_item(n);
      for (int n = 0; n < nitems && ok; ++n) {
        int j, w;
        tile_of(n, j, w);
        if (j > v_seen) {
          if (!(ok = wait_all(&v_full[j % NS], (j / NS) & 1))) break;
          v_seen = j;
        }
        if (!(ok = issue_pv(w, j, j % NS, n % 3, (n / 3) & 1))) break;
        if (n == last_item(j)) umma_commit_warp(&v_empty[j % NS]);
        if (n + 3 < nitems && !(ok = s_item(n + 3))) break;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;             // query tile of this warpgroup (a single-tile CTA: key tile parity)
    const int row = threadIdx.x & 127;    // tile row == TMEM lane
    const int rw = single ? r0 + half * kBlockM : r0 + wg * kBlockM;
    const int i = rw + row;
    const int my_nkv = wg ? nkv1 : nkv0;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + kOCol + wg * kOStride + lane_off;
    const int row_lim = CAUSAL ? min(Nk, i + 1) : Nk;  // admissible keys: [0, row_lim)
    const float2 sl2v = make_float2(sl2, sl2);
    float m_ref = -INFINITY;  // reference maximum, log2 units of the scaled score
    float dsum = 0.f;
    // O_w *= alpha (the caller has found a row of the warp that rescales).
    // O_w must hold exactly P_0..P_{j-1} first; completions of
    // O_w += P_w V are observed in order.  With two slots the landing of
    // S_j already implies that (its commit follows the issue of every
    // earlier product), so the wait returns at once, and a tile that does
    // not rescale does not wait at all.  With rotating slots this tile's
    // scores may be ready before the previous tile's product is even
    // issued; parity waits on the alternating barriers are exact: the
    // product two before (j - 3) has completed -- the commit of this tile's
    // S follows the issue of every product up to three items back -- and
    // the one after (j + 1) cannot start before this tile's P is released.
    // The rescale itself is rare (lazy), except on sharply peaked rows
    // whose maximum keeps growing.  64 columns per TMEM round trip.
    auto rescale_o = [&](int j, float alpha) -> bool {
      const bool w_ok =
          SLOTS == 3 ? mbar_wait(&o_done[2 * wg + ((j - 1) & 1)], ((j - 1) >> 1) & 1, wc, ATTN_ETIMEOUT)
                     : mbar_wait(&o_done[wg], (j - 1) & 1, wc, ATTN_ETIMEOUT);
      if (!__all_sync(0xffffffffu, w_ok)) return false;
      tc_fence_after();
      const float2 al = make_float2(alpha, alpha);
#pragma unroll
      for (int c = 0; c < HD / 32; c += 2) {
        uint32_t o2[2][32];
        tmem_ld32(tO + c * 32, o2[0]);
        tmem_ld32(tO + (c + 1) * 32, o2[1]);
        tmem_ld_wait(o2[0]);
        tmem_ld_wait(o2[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o2[h][e]), __uint_as_float(o2[h][e + 1])), al);
            o2[h][e] = __float_as_uint(v.x);
            o2[h][e + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tO + (c + h) * 32, o2[h]);
        }
      }
      return true;
    };
    bool ok = true;
    for (int j = 0; j < my_nkv; ++j) {
      // This tile's score slot and the parity of its use (see the item
      // numbering above; with two slots, slot = query tile).
      const int n = SLOTS == 3 ? (j < mmin ? 2 * j + wg : 2 * mmin + (j - mmin)) : j;
      const int slot = SLOTS == 3 ? n % 3 : wg;
      const uint32_t par = SLOTS == 3 ? (n / 3) & 1 : j & 1;
      const uint32_t tS = tmem + slot * 128 + lane_off;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[slot], par, wc, ATTN_ETIMEOUT));
      if (!ok) break;
      tc_fence_after();
      const int key0 = (t0 + (single ? 2 * j + wg : j)) * kBlockN;
      const bool masked = (key0 + kBlockN > Nk) || (CAUSAL && key0 + kBlockN - 1 > rw);
      const int lim = row_lim - key0;  // columns [0, lim) of this tile are admissible
      // The reducing TMEM load hands back each row's maximum with its
      // scores, so unmasked tiles need no maximum pass over the registers.
      // Masked columns must not enter the maximum: masked tiles (the
      // diagonal, the ragged last tile) mask and take a 3-input max pass.
      uint32_t sr[4][32];
      float m4[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + c * 32, sr[c], m4[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait_max(sr[c], m4[c]);
      float mx = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      if (masked) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e >= lim) sr[c][e] = __float_as_uint(-INFINITY);
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 8)
#pragma unroll
            for (int a = 0; a < 4; ++a)
              mx4[a] = max3(mx4[a], __uint_as_float(sr[c][e + 2 * a]), __uint_as_float(sr[c][e + 2 * a + 1]));
        mx = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
      }
      const float mt = (mx == -INFINITY) ? -INFINITY : mx * sl2;
      const bool resc = mt > m_ref + kTau;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_ref - mt);  // 0 on the first tile (m_ref = -inf)
        m_ref = mt;
        dsum *= alpha;
      }
      bool mid_ok = true;
      auto mid = [&]() {
        if constexpr (SPLIT_P == 2) {
          // Between the halves the first half's scores are dead and the
          // second half's are still in TMEM (P covers columns [0, 64) of
          // the slot): a rescaling warp drops them from registers for the
          // rescale and loads them back.
          if (j >= 1 && __any_sync(0xffffffffu, resc)) {
            mid_ok = rescale_o(j, alpha);
            if (mid_ok) {
              tmem_ld32(tS + 64, sr[2]);
              tmem_ld32(tS + 96, sr[3]);
              tmem_ld_wait(sr[2]);
              tmem_ld_wait(sr[3]);
              if (masked) {
#pragma unroll
                for (int c = 2; c < 4; ++c)
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    if (c * 32 + e >= lim) sr[c][e] = __float_as_uint(-INFINITY);
              }
            }
          }
        }
      };
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const float2 nm = make_float2(neg_m, neg_m);

      // p = 2^(s*sl2 - m_ref), written back over S as fp16 pairs (exp_row).
      // Masked and unmasked tiles run separate copies of the loop where that
      // was measured to pay (causal, D = 64); the non-causal D = 128 kernel
      // keeps one loop with the mask decided at run time.
      if constexpr (CAUSAL || HD == 64) {
        dsum += masked ? exp_row<2, EMU, SPLIT_P, FP8, HD == 64>(sr, sl2v, nm, true, lim, tS, &p_half[slot], &p_full[slot], mid)
                       : exp_row<1, EMU, SPLIT_P, FP8, HD == 64>(sr, sl2v, nm, false, lim, tS, &p_half[slot], &p_full[slot], mid);
      } else {
        dsum += exp_row<0, EMU, SPLIT_P, FP8, HD == 64>(sr, sl2v, nm, masked, lim, tS, &p_half[slot], &p_full[slot], mid);
      }
      if (!(ok = mid_ok)) break;
      if constexpr (!SPLIT_P) {
        if (j >= 1 && __any_sync(0xffffffffu, resc) && !(ok = rescale_o(j, alpha))) break;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[slot]);
      }
    }
    if constexpr (SLOTS == 3) {
      // the last two products, in order (each completion implies the ones before)
      for (int k = max(0, my_nkv - 2); k < my_nkv && ok; ++k)
        ok = __all_sync(0xffffffffu, mbar_wait(&o_done[2 * wg + (k & 1)], (k >> 1) & 1, wc, ATTN_ETIMEOUT));
    } else {
      if (ok && my_nkv > 0) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[wg], (my_nkv - 1) & 1, wc, ATTN_ETIMEOUT));
    }
    if (single && ok) {
      // ------------------------------------ single-tile CTA: merge, epilogue
      // Each warpgroup holds the carrier of its half of the key tiles for
      // the same 128 rows: (m_w, d_w) in registers, O_w in TMEM.  The carrier
      // merge: m = max(m0, m1), a_w = 2^(m_w - m), O = (a0 O0 + a1 O1) /
      // (a0 d0 + a1 d1).  The (m, d) pairs go through shared memory; then
      // warpgroup w finishes columns [w D/2, (w + 1) D/2) of every row,
      // reading them from both O accumulators (any warp may read the TMEM
      // lanes of its sub-partition, whichever warpgroup accumulated them).
      // The exchange overwrites the query tile, so each warpgroup first sees
      // both warpgroups' last products complete: their commits follow the
      // issue of every Q K^T (a warpgroup without a key tile has not waited
      // for any yet).
      if (nkv1 > 0 && wg == 0)
        ok = __all_sync(0xffffffffu, mbar_wait(&o_done[1], (nkv1 - 1) & 1, wc, ATTN_ETIMEOUT));
      if (wg == 1)
        ok = __all_sync(0xffffffffu, mbar_wait(&o_done[0], (nkv0 - 1) & 1, wc, ATTN_ETIMEOUT));
      if (ok) {
        x_m[wg * kBlockM + row] = m_ref;
        x_d[wg * kBlockM + row] = dsum;
        mbar_arrive(xchg);
        ok = __all_sync(0xffffffffu, mbar_wait(xchg, 0, wc, ATTN_ETIMEOUT));
        if (ok) {
          tc_fence_after();
          const float m0 = x_m[row], m1 = x_m[kBlockM + row];
          const float m = fmaxf(m0, m1);  // m0 is finite: warpgroup 0 always has a key tile
          const float a0 = ex2_approx(m0 - m);
          const float a1 = nkv1 > 0 ? ex2_approx(m1 - m) : 0.f;
          const float d = a0 * x_d[row] + a1 * x_d[kBlockM + row];
          const float inv = o_scale / d;  // o_scale: the E4M3 kernel's V descale, else 1
          const float2 c0 = make_float2(a0 * inv, a0 * inv), c1 = make_float2(a1 * inv, a1 * inv);
          const uint32_t tO0 = tmem + kOCol + lane_off, tO1 = tmem + kOCol + kOStride + lane_off;
          // O as fp16 into the first K/V stages (free: every product has
          // completed), in the 128B-swizzled layout of the 64-column TMA box:
          // at D = 128 warpgroup w fills box w, at D = 64 the two warpgroups
          // fill the halves of one box.  Rows past Nq are not stored.
          uint8_t* so = sK;
#pragma unroll
          for (int cc = 0; cc < HD / 64; ++cc) {
            const int c = wg * (HD / 64) + cc;  // this warpgroup's 32-column chunks
            uint32_t o0[32], o1[32];
            tmem_ld32(tO0 + c * 32, o0);
            if (nkv1 > 0) tmem_ld32(tO1 + c * 32, o1);
            tmem_ld_wait(o0);
            if (nkv1 > 0) {
              tmem_ld_wait(o1);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o1[e] = 0u;
            }
            uint32_t h[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 v = __ffma2_rn(make_float2(__uint_as_float(o1[2 * e]), __uint_as_float(o1[2 * e + 1])), c1,
                                          __fmul2_rn(make_float2(__uint_as_float(o0[2 * e]), __uint_as_float(o0[2 * e + 1])), c0));
              h[e] = pack_half2(v.x, v.y);
            }
            uint8_t* srow = so + (c >> 1) * kChunkBytes + row * 128;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int u = (c & 1) * 4 + e;
              *reinterpret_cast<uint4*>(srow + ((u ^ (row & 7)) << 4)) =
                  make_uint4(h[4 * e], h[4 * e + 1], h[4 * e + 2], h[4 * e + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&o_staged[wg]);
          if (row == 0 && (HD == 128 || wg == 0)) {
            bool staged = mbar_wait(&o_staged[wg], 0, wc, ATTN_ETIMEOUT);
            if (HD == 64 && staged) staged = mbar_wait(&o_staged[1], 0, wc, ATTN_ETIMEOUT);
            if (staged) {
              tma_store_3d(&tmO, so + wg * kChunkBytes, 64 * wg, rw, bh);
              bulk_commit_group();
              bulk_wait_read_all();
            }
          }
          if (wg == 0 && lse != nullptr && i < Nq)
            lse[static_cast<size_t>(bh) * Nq + i] = (m + log2f(d)) * 0.69314718055994531f;
        }
      }
    } else if (ok && my_nkv > 0 && !SPLITKV) {
      // ---------------------------------------------------------- epilogue
      tc_fence_after();
      const float inv = o_scale / dsum;  // o_scale: the E4M3 kernel's V descale, else 1
      const float2 iv = make_float2(inv, inv);
      if constexpr (!FP8) {
        // O / d as fp16 into this warpgroup's query-tile buffer (free: every
        // Q_w K^T was issued before the last O_w += P_w V, whose completion
        // was just seen), in the 128B-swizzled layout of the TMA box --
        // 16-byte unit u of row r at u ^ (r mod 8) -- then one thread
        // stores the tile with TMA; rows past Nq lie outside the tensor and
        // are not written.
        uint8_t* so = sQ + wg * TB;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tO + c * 32, orr);
          tmem_ld_wait(orr);
          uint32_t h[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1])), iv);
            h[e] = pack_half2(v.x, v.y);
          }
          uint8_t* srow = so + (c >> 1) * kChunkBytes + row * 128;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int u = (c & 1) * 4 + e;
            *reinterpret_cast<uint4*>(srow + ((u ^ (row & 7)) << 4)) =
                make_uint4(h[4 * e], h[4 * e + 1], h[4 * e + 2], h[4 * e + 3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&o_staged[wg]);
        if (row == 0) {
          if (mbar_wait(&o_staged[wg], 0, wc, ATTN_ETIMEOUT)) {
#pragma unroll
            for (int k = 0; k < HD / 64; ++k) tma_store_3d(&tmO, so + k * kChunkBytes, k * 64, rw, bh);
            bulk_commit_group();
            bulk_wait_read_all();
          }
        }
      } else {
        __half* orow = out + (static_cast<size_t>(bh) * Nq + i) * HD;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tO + c * 32, orr);
          tmem_ld_wait(orr);
          if (i < Nq) {
            uint32_t h[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1])), iv);
              h[e] = pack_half2(v.x, v.y);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(h[4 * e], h[4 * e + 1], h[4 * e + 2], h[4 * e + 3]);
          }
        }
      }
      if (lse != nullptr && i < Nq)
        lse[static_cast<size_t>(bh) * Nq + i] = (m_ref + log2f(dsum)) * 0.69314718055994531f;
    }
    if (ok && SPLITKV) {
      // ------------------------------------------- split-KV part epilogue
      // This share's carrier, normalised: O_s = o / d in fp32 and its
      // log-sum-exp in log2 units (-inf when the share has no admissible key
      // for this tile); the merge kernel combines the shares.
      if (my_nkv > 0) tc_fence_after();
      const float inv = my_nkv > 0 ? 1.f / dsum : 0.f;
      const size_t rr = static_cast<size_t>(blockIdx.z) * rows_total + static_cast<size_t>(bh) * Nq + i;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t orr[32];
        if (my_nkv > 0) {
          tmem_ld32(tO + c * 32, orr);
          tmem_ld_wait(orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        if (i < Nq) {
          float4* dst = reinterpret_cast<float4*>(ws_o + rr * HD + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(orr[4 * e]) * inv, __uint_as_float(orr[4 * e + 1]) * inv,
                                 __uint_as_float(orr[4 * e + 2]) * inv, __uint_as_float(orr[4 * e + 3]) * inv);
        }
      }
      if (i < Nq) ws_l[rr] = my_nkv > 0 ? m_ref + log2f(dsum) : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out somewhere in this CTA: let every TMA copy and every
    // tensor-core op it issued land before the shared memory and TMEM go.
    if (warp == kProducerWarp && lane == 0) {
      mbar_wait(q_full, 0, wc, ATTN_ETIMEOUT, false);
      for (int s = 0; s < NS; ++s) {
        if (last_k[s] >= 0) mbar_wait(&k_full[s], (last_k[s] / NS) & 1, wc, ATTN_ETIMEOUT, false);
        if (last_v[s] >= 0) mbar_wait(&v_full[s], (last_v[s] / NS) & 1, wc, ATTN_ETIMEOUT, false);
      }
    }
    if (warp == kMmaWarp) {
      umma_commit_warp(drain);
      mbar_wait(drain, 0, wc, ATTN_ETIMEOUT, false);
      __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // A single-tile launch that may have started next to the pairs' launch
  // (see launch_kernel) ends only after that grid has completed, so the
  // forward as a whole completes in stream order (no-op otherwise).
  if constexpr (SINGLE) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Merge of the split-KV parts: the carrier merge of partial states
// (m1,d1,o1) (+) (m2,d2,o2), applied to normalised parts.  For one row, with
// l_s each part's log-sum-exp in log2 units and O_s its normalised output,
//   m = max_s l_s,  w_s = 2^(l_s - m),  O = sum_s w_s O_s / sum_s w_s,
//   LSE = ln2 * (m + log2 sum_s w_s).
// An empty part has l_s = -inf and weight 0.  One warp per row; lane t owns
// HD/32 consecutive columns, so every load of a part's row is coalesced.
template <int HD>
__global__ void __launch_bounds__(128)
attn_splitkv_merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_l,
                          __half* __restrict__ out, float* __restrict__ lse, size_t rows, int splits) {
  constexpr int kPer = HD / 32;
  const size_t row = static_cast<size_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // Launched as a programmatic dependent of the split forward: wait for
  // that grid to complete and its parts to be visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Like the forward, no work while the status word holds an error: the
  // parts of a forward that stopped early were never written.
  if (*static_cast<volatile int*>(&g_attn_status) != 0) return;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, ws_l[static_cast<size_t>(s) * rows + row]);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const size_t rr = static_cast<size_t>(s) * rows + row;
      const float w = ex2_approx(ws_l[rr] - m);
      den += w;
      const float* src = ws_o + rr * HD + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
        acc[2] += w * x.z;
        acc[3] += w * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __half* dst = out + row * HD + lane * kPer;
  if constexpr (kPer == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_half2(acc[0] * inv, acc[1] * inv), pack_half2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_half2(acc[0] * inv, acc[1] * inv);
  }
  if (lse != nullptr && lane == 0) lse[row] = den > 0.f ? (m + log2f(den)) * 0.69314718055994531f : -INFINITY;
}

// V^T for the E4M3 kernel, whose O += P V takes V K-major (keys contiguous):
// vt[bh][d][key] = v[bh][key][d] for D = 128, rows of ldk bytes (the key
// count rounded up to 16; the keys in between are written as zero).  One CTA
// per 128 keys of one head: the tile goes through shared memory as 32-bit
// words (rows padded to 33 words, so that both phases are free of bank
// conflicts), and each thread turns four 4 x 4 byte blocks around with byte
// permutes into 16 consecutive keys of 4 rows of V^T.
__global__ void __launch_bounds__(256)
attn_fp8_transpose_v_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt, int Nk, int ldk) {
  __shared__ uint32_t tile[128][33];
  const size_t bh = blockIdx.y;
  const int k0 = blockIdx.x * 128;
  const uint8_t* src = v + bh * static_cast<size_t>(Nk) * 128;
  for (int c = threadIdx.x; c < 1024; c += blockDim.x) {
    const int key = c >> 3, part = c & 7;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + key < Nk) val = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(k0 + key) * 128 + part * 16);
    tile[key][4 * part] = val.x;
    tile[key][4 * part + 1] = val.y;
    tile[key][4 * part + 2] = val.z;
    tile[key][4 * part + 3] = val.w;
  }
  __syncthreads();
  const int db = threadIdx.x & 31;  // rows 4 db .. 4 db + 3 of V^T
  const int kb = threadIdx.x >> 5;  // keys k0 + 16 kb .. + 15
  if (k0 + 16 * kb >= ldk) return;
  uint32_t out[4][4];  // [row j][group g]: keys 4g .. 4g + 3 of row 4 db + j
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int r = 16 * kb + 4 * g;
    const uint32_t w0 = tile[r][db], w1 = tile[r + 1][db], w2 = tile[r + 2][db], w3 = tile[r + 3][db];
    const uint32_t a = __byte_perm(w0, w1, 0x5140), b = __byte_perm(w2, w3, 0x5140);  // bytes 0, 1
    const uint32_t c = __byte_perm(w0, w1, 0x7362), d = __byte_perm(w2, w3, 0x7362);  // bytes 2, 3
    out[0][g] = __byte_perm(a, b, 0x5410);
    out[1][g] = __byte_perm(a, b, 0x7632);
    out[2][g] = __byte_perm(c, d, 0x5410);
    out[3][g] = __byte_perm(c, d, 0x7632);
  }
  uint8_t* dst = vt + bh * 128 * static_cast<size_t>(ldk) + k0 + 16 * kb;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(4 * db + j) * ldk) =
        make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
}

// The softmax's E4M3 packing on its own, for tests: out[i] packs in[4i..4i+3].
__global__ void attn_debug_pack_e4m3_kernel(const float* __restrict__ in, uint32_t* __restrict__ out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = pack_e4m3x4(in[4 * i], in[4 * i + 1], in[4 * i + 2], in[4 * i + 3]);
}

// 2^x on the FMA pipe (exp2_poly2) on its own, for tests: out[i] = 2^in[i].
__global__ void attn_debug_exp2_poly_kernel(const float* __restrict__ in, float* __restrict__ out, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float2 x = make_float2(in[i], i + 1 < n ? in[i + 1] : in[i]);
  const float2 y = exp2_poly2(x);
  out[i] = y.x;
  if (i + 1 < n) out[i + 1] = y.y;
}

// =====================================================================
// Host side
// =====================================================================
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
uint64_t g_timeout_ns = kDefaultTimeoutNs;
int g_drop_tile = -1;
constexpr int kMaxDevices = 64;

// A driver entry point, looked up through the runtime (so that the library
// loads on a machine without a driver).  Call with g_mu held.
template <typename Fn>
Fn driver_fn(const char* name) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(fn);
}

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) g_encode = driver_fn<EncodeTiledFn>("cuTensorMapEncodeTiled");
  return g_encode;
}

// [BH, N, D] fp16 viewed as a 3-D tensor (D innermost); box = 64 x 128 x 1
// with the 128-byte swizzle.  Rows past N read as zero.
bool make_map(CUtensorMap* m, const void* base, int64_t BH, int64_t N, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(N) * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 tensors as bytes: [BH, rows, cols] with row stride ld (a multiple of
// 16 bytes); box = 128 x 128 x 1 with the 128-byte swizzle.  Elements past
// cols or rows read as zero.
bool make_map_u8(CUtensorMap* m, const void* base, int64_t BH, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld), static_cast<cuuint64_t>(rows * ld)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// ------------------------------------------------------------ device state
// Built-in scratch of attn_fwd_splitkv_noalloc: holds the split-KV parts for
// callers that cannot allocate device memory.  Every device that loads the
// library carries it until the process exits.  In host code the name below
// only stands in for the buffer; its device address comes from
// cudaGetSymbolAddress, looked up with the device current (ContextState).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(ATTN_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// What the library keeps per CUDA context: the sm_103 check and SM count,
// the host copy of the device status word (page-locked host memory mapped
// into the device: kernels write it when a wait runs out, and the entry
// points read it before enqueueing anything), and the device address of the
// no-allocation scratch.  Entries are keyed by the context's unique id: a
// context reset (cudaDeviceReset) makes a new context, whose first call
// sets up a new entry, while the old entry's memory went with the old
// context.  Created on the first call in a context and never freed.
struct ContextState {
  unsigned long long ctx_id = 0;
  int sms = 0;                    // > 0, or 0 when the device is not an sm_103 part
  int* status_host = nullptr;     // host view of the copy (null if it could not be made)
  int* status_dev = nullptr;      // device view of the same word
  void* noalloc = nullptr;        // device address of g_noalloc_scratch (looked up on first use)
};
constexpr int kMaxContexts = 64;
ContextState g_ctx[kMaxContexts];
int g_nctx = 0;

// Unique id of the calling thread's current context (made current by the
// runtime if none is).  Call with g_mu held.
bool current_ctx_id(unsigned long long* id) {
  if (!g_ctx_current) g_ctx_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  if (!g_ctx_id) g_ctx_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) {  // the runtime has not bound its primary context to this thread yet
    if (cudaFree(nullptr) != cudaSuccess || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  }
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// The current context's entry, created on first use; call with g_mu held.
// Returns ATTN_OK, ATTN_EUNSUPPORTED (not an sm_103 part) or ATTN_ECUDA.
int context_state(ContextState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ECUDA;
  unsigned long long id = 0;
  if (!current_ctx_id(&id)) return ATTN_ECUDA;
  ContextState* st = nullptr;
  for (int i = 0; i < g_nctx && !st; ++i)
    if (g_ctx[i].ctx_id == id) st = &g_ctx[i];
  if (!st) {
    ContextState fresh;
    fresh.ctx_id = id;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_ECUDA;
    fresh.sms = (prop.major == 10 && prop.minor == 3) ? prop.multiProcessorCount : 0;
    if (fresh.sms > 0) {
      int* h = nullptr;
      void* d = nullptr;
      if (cudaHostAlloc(reinterpret_cast<void**>(&h), sizeof(int), cudaHostAllocMapped | cudaHostAllocPortable) ==
          cudaSuccess) {
        if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) {
          *h = 0;
          fresh.status_host = h;
          fresh.status_dev = static_cast<int*>(d);
        } else {
          cudaFreeHost(h);
        }
      }
      cudaGetLastError();  // a failed optional step leaves no sticky runtime error behind
    }
    if (g_nctx == kMaxContexts) {  // table full (many contexts): serve without caching
      static thread_local ContextState spare;
      spare = fresh;
      st = &spare;
    } else {
      g_ctx[g_nctx] = fresh;
      st = &g_ctx[g_nctx++];
    }
  }
  if (st->sms <= 0) return ATTN_EUNSUPPORTED;
  *out = st;
  return ATTN_OK;
}

// What every launch takes besides its tensors: the host copy of the status
// word and the testing hook's settings.
struct RunCtl {
  int* status_dev = nullptr;
  uint64_t timeout_ns = kDefaultTimeoutNs;
  int drop = -1;
  int sms = 0;
  void* noalloc = nullptr;
};

// Entry of every forward call (after its argument checks): the current
// context's state and the testing hook's settings.  Returns ATTN_ETIMEOUT,
// without touching the device, while the host copy of the status word holds
// an error that attn_get_status() has not yet cleared.  want_noalloc also
// looks up the no-allocation scratch (once per context).
int enter(RunCtl* rc, bool want_noalloc = false) {
  std::lock_guard<std::mutex> lk(g_mu);
  ContextState* st = nullptr;
  const int r = context_state(&st);
  if (r != ATTN_OK) return r;
  if (st->status_host != nullptr && *static_cast<volatile int*>(st->status_host) != 0) return ATTN_ETIMEOUT;
  if (want_noalloc && st->noalloc == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ECUDA;
    st->noalloc = ptr;
  }
  rc->status_dev = st->status_dev;
  rc->timeout_ns = g_timeout_ns;
  rc->drop = g_drop_tile;
  rc->sms = st->sms;
  rc->noalloc = st->noalloc;
  return ATTN_OK;
}

// ------------------------------------------------------------ launches
template <int HD, bool CAUSAL, int NS, int SPLIT_P, int EMU, bool SPLITKV, bool FP8 = false, int SLOTS = 2,
          bool SINGLE = false>
int launch_kernel(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                  void* o, float* lse,
                  float* ws_o, float* ws_l, dim3 grid, int Nq, int Nk, float sl2, int n_main, cudaStream_t st,
                  const RunCtl& rc, float o_scale, bool after_pairs = false) {
  using L = Layout<HD, NS, FP8, SINGLE ? 1 : 2>;
  auto kern = attn_fwd_kernel<HD, CAUSAL, NS, SPLIT_P, EMU, SPLITKV, FP8, SLOTS, SINGLE>;
  static_assert(L::kSmem <= 232448, "shared memory budget");
  // The shared-memory attribute is set on the first launch on each device
  // only: the host-buffer entry points launch once per chunk, and every
  // driver call there is on the path that keeps the GPU fed.
  static std::atomic<uint64_t> attr_set{0};  // one bit per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ECUDA;
  const uint64_t bit = 1ull << dev;
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kSmem)) !=
        cudaSuccess)
      return ATTN_ECUDA;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  // The single-tile launch that follows a launch of pairs may start while
  // the pairs' last wave still runs (programmatic dependent launch): its
  // CTAs take SMs as they free up instead of after the slowest pair CTA
  // and a launch gap.  The two grids touch disjoint rows, and each
  // single-tile CTA waits for the pairs' grid before it exits, so work
  // after the forward on the stream still follows all of it.
  auto launch = [&]() -> cudaError_t {
    if (!after_pairs) {
      kern<<<grid, kThreads, L::kSmem, st>>>(mq, mk, mv, mo, static_cast<__half*>(o), lse, ws_o, ws_l, Nq, Nk, sl2,
                                             o_scale, rc.status_dev, rc.timeout_ns, rc.drop, n_main);
      return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, static_cast<__half*>(o), lse, ws_o, ws_l, Nq, Nk, sl2,
                              o_scale, rc.status_dev, rc.timeout_ns, rc.drop, n_main);
  };
  if (launch() == cudaSuccess) return ATTN_OK;
  cudaGetLastError();
  // A context reset (cudaDeviceReset) drops the attribute: set it again and
  // retry once (a launch that failed did not run).
  attr_set.fetch_and(~bit, std::memory_order_acq_rel);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kSmem)) !=
      cudaSuccess)
    return ATTN_ECUDA;
  attr_set.fetch_or(bit, std::memory_order_release);
  return launch() == cudaSuccess ? ATTN_OK : ATTN_ECUDA;
}

// One forward: the grid of (query-tile pair, head, share) CTAs.  For the
// single pass (fp16 or E4M3), the pairs of a last partial wave that would
// occupy at most half the SMs go to a second launch of single-tile CTAs
// (two per pair, half the work each), which runs as soon as the full waves
// are done: that wave then takes half as long (causal: grids of at most one
// wave of pairs only, as one launch of single-tile CTAs).
// Pairs of the last partial wave that go to single-tile CTAs: all of the
// last wave's pairs when it would occupy at most half of the `sms` SMs --
// and, when full waves of pairs come first, only if each query tile has at
// least 16 key tiles: the second launch then waits for the full waves and
// costs a few microseconds, more than half a wave of short CTAs saves.
// Causal: only a whole grid of at most one wave of pairs, which then runs
// as single-tile CTAs alone, heaviest first (up to two waves of them: the
// light tiles of the triangle fill the second).  Larger causal grids keep
// their pairs, ordered heaviest first, whose last wave holds the lightest.
// Non-causal grids whose pairs are often half empty (a query length that
// leaves the second tile of a head's last pair past Nq) also run as
// single-tile CTAs alone when that takes clearly fewer waves: a single-tile
// CTA costs about 0.65 of a pair CTA over the same key tiles (measured
// 0.57-0.6 on long key ranges), and only the query tiles that exist cost
// anything.  `q_tiles` counts those over all heads.
int64_t tail_pairs(int64_t pairs, int sms, int key_tiles, bool causal, int64_t q_tiles) {
  if (sms <= 0) return 0;
  if (causal) return pairs <= sms ? pairs : 0;
  const int64_t last = pairs % sms;
  int64_t tail = last;
  if (last == 0 || 2 * last > sms || (last < pairs && key_tiles < 16)) tail = 0;
  const double waves_now = static_cast<double>((pairs - tail + sms - 1) / sms) + (tail > 0 ? 0.65 : 0.0);
  const double waves_single = 0.65 * static_cast<double>((q_tiles + sms - 1) / sms);
  if (waves_single < 0.9 * waves_now) return pairs;
  return tail;
}

template <int HD, bool CAUSAL, int NS, int SPLIT_P, int EMU, bool SPLITKV, bool FP8 = false, int SLOTS = 2>
int launch_fwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
               void* o, float* lse,
               float* ws_o, float* ws_l, int BH, int Nq, int Nk, float sl2, int splits, cudaStream_t st,
               const RunCtl& rc, float o_scale = 1.0f) {
  const int n_pairs = (Nq + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t pairs = static_cast<int64_t>(n_pairs) * BH;
  constexpr bool kTail = !SPLITKV;
  const int64_t q_tiles = static_cast<int64_t>(BH) * ((Nq + kBlockM - 1) / kBlockM);
  const int64_t tail = kTail ? tail_pairs(pairs, rc.sms, (Nk + kBlockN - 1) / kBlockN, CAUSAL, q_tiles) : 0;
  if (pairs > 0x7fffffff) return ATTN_EUNSUPPORTED;
  const int n_main = static_cast<int>(pairs - tail);
  if (n_main > 0) {
    const int r = launch_kernel<HD, CAUSAL, NS, SPLIT_P, EMU, SPLITKV, FP8, SLOTS, false>(
        mq, mk, mv, mo, o, lse, ws_o, ws_l, dim3(n_pairs, BH, splits), Nq, Nk, sl2, n_main, st, rc, o_scale);
    if (r != ATTN_OK) return r;
  }
  if constexpr (kTail) {
    // The single-tile CTAs use two score slots, one per warpgroup, also at
    // D = 64 (their warpgroups alternate key tiles, so slots need not rotate).
    if (tail > 0)
      return launch_kernel<HD, CAUSAL, single_stages<HD, FP8>(), SPLIT_P, EMU, SPLITKV, FP8, 2, true>(
          mq, mk, mv, mo, o, lse, ws_o, ws_l, dim3(static_cast<unsigned>(2 * tail)), Nq, Nk, sl2, n_main, st, rc,
          o_scale, n_main > 0);
  }
  return ATTN_OK;
}

// The fp16 forward: D = 64 with three rotating score slots and P released
// whole, D = 128 with P released in two halves.  EMU: one pair of
// exponentials in EMU on the FMA-pipe polynomial (0 = none).
template <bool SPLITKV, int EMU64 = kEmu64, int EMU128 = kEmu128>
int dispatch_fwd(int D, int causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                 const CUtensorMap& mo, void* o, float* lse, float* ws_o, float* ws_l, int BH, int Nq, int Nk, float sl2, int splits,
                 cudaStream_t st, const RunCtl& rc) {
  if (D == 64)
    return causal ? launch_fwd<64, true, 4, 0, EMU64, SPLITKV, false, 3>(mq, mk, mv, mo, o, lse, ws_o, ws_l, BH, Nq, Nk,
                                                                         sl2, splits, st, rc)
                  : launch_fwd<64, false, 4, 0, EMU64, SPLITKV, false, 3>(mq, mk, mv, mo, o, lse, ws_o, ws_l, BH, Nq, Nk,
                                                                          sl2, splits, st, rc);
  return causal ? launch_fwd<128, true, 2, 2, EMU128, SPLITKV>(mq, mk, mv, mo, o, lse, ws_o, ws_l, BH, Nq, Nk, sl2,
                                                               splits, st, rc)
                : launch_fwd<128, false, 2, 2, EMU128, SPLITKV>(mq, mk, mv, mo, o, lse, ws_o, ws_l, BH, Nq, Nk, sl2,
                                                                splits, st, rc);
}

// Argument checks shared by the forward entry points (no CUDA call).
// Returns ATTN_OK with *empty set when there is nothing to compute.
int check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H,
               int Nq, int Nk, int D, float scale, bool* empty) {
  *empty = false;
  if (!q || !k || !v || !o) return ATTN_EINVAL;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 1) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_EINVAL;
  if (D != 64 && D != 128) return ATTN_EUNSUPPORTED;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_EUNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 65535) return ATTN_EUNSUPPORTED;
  if (B == 0 || H == 0 || Nq == 0) {
    *empty = true;
    return ATTN_OK;
  }
  const int BH = B * H;
  const size_t qbytes = static_cast<size_t>(BH) * Nq * D * 2, kvbytes = static_cast<size_t>(BH) * Nk * D * 2;
  if (ranges_overlap(o, qbytes, q, qbytes) || ranges_overlap(o, qbytes, k, kvbytes) ||
      ranges_overlap(o, qbytes, v, kvbytes))
    return ATTN_EUNSUPPORTED;
  const size_t lbytes = static_cast<size_t>(BH) * Nq * 4;
  if (lse && (ranges_overlap(lse, lbytes, o, qbytes) || ranges_overlap(lse, lbytes, q, qbytes) ||
              ranges_overlap(lse, lbytes, k, kvbytes) || ranges_overlap(lse, lbytes, v, kvbytes)))
    return ATTN_EUNSUPPORTED;
  return ATTN_OK;
}

// Key tiles of the longest query-tile pair (the kernel's nkv for the pair
// with the most admissible keys).
int64_t pair_key_tiles(int Nq, int Nk, int causal) {
  const int64_t pairs_end = (static_cast<int64_t>(Nq) + kRowsPerCta - 1) / kRowsPerCta * kRowsPerCta;
  const int64_t keys = causal ? std::min<int64_t>(Nk, pairs_end) : Nk;
  return (keys + kBlockN - 1) / kBlockN;
}

// ATTN_ETOOLONG when a row would accumulate more than ATTN_MAX_KEYS_PER_PASS
// keys in one pass (one share of `splits`); 0 = the single-pass forward.
int check_keys_per_pass(int Nq, int Nk, int causal, int splits) {
  if (splits == 0) {
    const int64_t keys = causal ? std::min(Nk, Nq) : Nk;
    return keys > ATTN_MAX_KEYS_PER_PASS ? ATTN_ETOOLONG : ATTN_OK;
  }
  const int64_t share_tiles = (pair_key_tiles(Nq, Nk, causal) + splits - 1) / splits;
  return share_tiles * kBlockN > ATTN_MAX_KEYS_PER_PASS ? ATTN_ETOOLONG : ATTN_OK;
}

constexpr int kMaxSplits = 256;

size_t splitkv_bytes(int B, int H, int Nq, int D, int splits) {
  return static_cast<size_t>(splits) * B * H * Nq * (D + 1) * sizeof(float);
}

template <int HD>
int launch_merge(const float* ws_o, const float* ws_l, void* o, float* lse, size_t rows, int splits,
                 cudaStream_t st) {
  const size_t blocks = (rows + 3) / 4;
  if (blocks > 0x7fffffffu) return ATTN_EUNSUPPORTED;
  // A programmatic dependent launch: the merge's CTAs are placed while the
  // split forward's last CTAs still run, and wait for its grid in the kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_splitkv_merge_kernel<HD>, ws_o, ws_l,
                                           static_cast<__half*>(o), lse, rows, splits);
  return e == cudaSuccess ? ATTN_OK : ATTN_ECUDA;
}

// The split-KV forward and its merge on `workspace` (parts, then the
// per-row log-sum-exps), once the arguments have been checked.
int enqueue_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int Nq, int Nk, int D,
                    float scale, int causal, int num_splits, void* workspace, cudaStream_t st, const RunCtl& rc) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, BH, Nq, D) || !make_map(&mk, k, BH, Nk, D) || !make_map(&mv, v, BH, Nk, D))
    return ATTN_ECUDA;
  const float sl2 = scale * 1.4426950408889634f;
  const size_t rows = static_cast<size_t>(BH) * Nq;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_l = ws_o + static_cast<size_t>(num_splits) * rows * D;
  // (the split-KV parts write fp32 carriers, not O: the O map is unused)
  const int r = dispatch_fwd<true>(D, causal, mq, mk, mv, mq, o, lse, ws_o, ws_l, BH, Nq, Nk, sl2, num_splits, st, rc);
  if (r != ATTN_OK) return r;
  return D == 64 ? launch_merge<64>(ws_o, ws_l, o, lse, rows, num_splits, st)
                 : launch_merge<128>(ws_o, ws_l, o, lse, rows, num_splits, st);
}

// Streams and events of attn_fwd_host, created once per device on first
// use (never per call) and kept until the process exits.  One mutex guards
// the enqueue, so calls from several host threads serialise on them.
constexpr int kMaxHostChunks = 64;
struct HostPipe {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_comp[2] = {nullptr, nullptr}, s_out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in[kMaxHostChunks] = {}, comp[kMaxHostChunks] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

HostPipe* host_pipe(int dev) {  // call with g_pipe_mu held
  HostPipe& p = g_pipe[dev];
  if (p.ready) return &p;
  const unsigned f = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.s_comp[0], cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.s_comp[1], cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&p.start, f) == cudaSuccess && cudaEventCreateWithFlags(&p.done, f) == cudaSuccess;
  for (int c = 0; ok && c < kMaxHostChunks; ++c)
    ok = cudaEventCreateWithFlags(&p.in[c], f) == cudaSuccess && cudaEventCreateWithFlags(&p.comp[c], f) == cudaSuccess;
  if (!ok) return nullptr;  // what was created stays for the next attempt to reuse or leak; rare
  p.ready = true;
  return &p;
}

// The chunked pipeline of the host-buffer entry points over the flattened
// B*H heads: chunk c's inputs are copied in on s_in, compute(c, h0, nb,
// stream) enqueues its forward on one of the two compute streams (taken in
// turn, so that the next chunk's CTAs take the SMs the current one frees in
// its last wave), and its outputs are copied out on s_out.  in_elem: bytes
// per Q/K/V element (O is fp16, LSE fp32).
template <typename Compute>
int host_pipeline(int dev, const void* q_host, const void* k_host, const void* v_host, void* o_host,
                  float* lse_host, void* q_dev, void* k_dev, void* v_dev, const void* o_dev, const float* lse_dev,
                  int BH, int Nq, int Nk, int D, int in_elem, int chunks, cudaStream_t user, Compute&& compute) {
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* p = host_pipe(dev);
  if (!p) return ATTN_ECUDA;
  // Every internal stream starts after the work already queued on `user`
  // (which may still use the device buffers), and `user` resumes when the
  // last output has reached host memory.
  if (cudaEventRecord(p->start, user) != cudaSuccess || cudaStreamWaitEvent(p->s_in, p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->s_comp[0], p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->s_comp[1], p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->s_out, p->start, 0) != cudaSuccess)
    return ATTN_ECUDA;
  const auto H2D = cudaMemcpyHostToDevice;
  const auto D2H = cudaMemcpyDeviceToHost;
  auto at = [](const void* b, size_t off) { return static_cast<const char*>(b) + off; };
  auto atw = [](void* b, size_t off) { return static_cast<char*>(b) + off; };
  for (int c = 0; c < chunks; ++c) {
    cudaStream_t sc = p->s_comp[c & 1];
    // heads [h0, h0 + nb): contiguous in every tensor
    const int h0 = static_cast<int>(static_cast<int64_t>(BH) * c / chunks);
    const int nb = static_cast<int>(static_cast<int64_t>(BH) * (c + 1) / chunks) - h0;
    const size_t qi = static_cast<size_t>(in_elem) * Nq * D, ki = static_cast<size_t>(in_elem) * Nk * D;
    const size_t oo = static_cast<size_t>(h0) * Nq * D * 2, on = static_cast<size_t>(nb) * Nq * D * 2;
    const size_t lo = static_cast<size_t>(h0) * Nq, ln = static_cast<size_t>(nb) * Nq * 4;
    if (cudaMemcpyAsync(atw(q_dev, h0 * qi), at(q_host, h0 * qi), nb * qi, H2D, p->s_in) != cudaSuccess ||
        cudaMemcpyAsync(atw(k_dev, h0 * ki), at(k_host, h0 * ki), nb * ki, H2D, p->s_in) != cudaSuccess ||
        cudaMemcpyAsync(atw(v_dev, h0 * ki), at(v_host, h0 * ki), nb * ki, H2D, p->s_in) != cudaSuccess ||
        cudaEventRecord(p->in[c], p->s_in) != cudaSuccess || cudaStreamWaitEvent(sc, p->in[c], 0) != cudaSuccess)
      return ATTN_ECUDA;
    const int r = compute(c, h0, nb, sc);
    if (r != ATTN_OK) return r;
    if (cudaEventRecord(p->comp[c], sc) != cudaSuccess || cudaStreamWaitEvent(p->s_out, p->comp[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(atw(o_host, oo), at(o_dev, oo), on, D2H, p->s_out) != cudaSuccess ||
        (lse_host && cudaMemcpyAsync(lse_host + lo, lse_dev + lo, ln, D2H, p->s_out) != cudaSuccess))
      return ATTN_ECUDA;
  }
  if (cudaEventRecord(p->done, p->s_out) != cudaSuccess || cudaStreamWaitEvent(user, p->done, 0) != cudaSuccess)
    return ATTN_ECUDA;
  return ATTN_OK;
}

// Argument checks of the E4M3 entry points (no CUDA call); *empty as check_args.
int check_args_fp8(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H,
                   int Nq, int Nk, int D, float scale, float q_descale, float k_descale, float v_descale,
                   const void* workspace, size_t workspace_bytes, bool* empty) {
  *empty = false;
  if (!q || !k || !v || !o) return ATTN_EINVAL;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 1) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_EINVAL;
  if (!std::isfinite(q_descale) || !std::isfinite(k_descale) || !std::isfinite(v_descale) || q_descale <= 0.f ||
      k_descale <= 0.f || v_descale <= 0.f)
    return ATTN_EINVAL;
  if (D != 128) return ATTN_EUNSUPPORTED;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_EUNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 65535) return ATTN_EUNSUPPORTED;
  if (B == 0 || H == 0 || Nq == 0) {
    *empty = true;
    return ATTN_OK;
  }
  const size_t need = static_cast<size_t>(B) * H * D * ((static_cast<size_t>(Nk) + 15) / 16 * 16);
  if (!workspace || workspace_bytes < need) return ATTN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return ATTN_EUNSUPPORTED;
  const int BH = B * H;
  const size_t qb = static_cast<size_t>(BH) * Nq * D, kb = static_cast<size_t>(BH) * Nk * D;
  const size_t ob = qb * 2, lb = static_cast<size_t>(BH) * Nq * 4;
  if (ranges_overlap(o, ob, q, qb) || ranges_overlap(o, ob, k, kb) || ranges_overlap(o, ob, v, kb) ||
      ranges_overlap(workspace, need, q, qb) || ranges_overlap(workspace, need, k, kb) ||
      ranges_overlap(workspace, need, v, kb) || ranges_overlap(workspace, need, o, ob))
    return ATTN_EUNSUPPORTED;
  if (lse && (ranges_overlap(lse, lb, o, ob) || ranges_overlap(lse, lb, q, qb) || ranges_overlap(lse, lb, k, kb) ||
              ranges_overlap(lse, lb, v, kb) || ranges_overlap(lse, lb, workspace, need)))
    return ATTN_EUNSUPPORTED;
  return ATTN_OK;
}

// Encodes the E4M3 forward's maps for heads [h0, h0 + nb) and enqueues the
// V transpose and the forward on `st`.
int enqueue_fp8(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace, int h0, int nb,
                int Nq, int Nk, float sl2, float v_descale, int causal, cudaStream_t st, const RunCtl& rc) {
  const int D = 128;
  const int ldk = (Nk + 15) / 16 * 16;
  const size_t qo = static_cast<size_t>(h0) * Nq * D, ko = static_cast<size_t>(h0) * Nk * D;
  const size_t wo = static_cast<size_t>(h0) * D * ldk;
  const uint8_t* qc = static_cast<const uint8_t*>(q) + qo;
  const uint8_t* kc = static_cast<const uint8_t*>(k) + ko;
  const uint8_t* vc = static_cast<const uint8_t*>(v) + ko;
  uint8_t* wc = static_cast<uint8_t*>(workspace) + wo;
  __half* oc = static_cast<__half*>(o) + qo;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map_u8(&mq, qc, nb, Nq, D, D) || !make_map_u8(&mk, kc, nb, Nk, D, D) ||
      !make_map_u8(&mv, wc, nb, D, Nk, ldk) || !make_map(&mo, oc, nb, Nq, D))
    return ATTN_ECUDA;
  attn_fp8_transpose_v_kernel<<<dim3((Nk + 127) / 128, nb), 256, 0, st>>>(vc, wc, Nk, ldk);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ECUDA;
  float* lc = lse ? lse + static_cast<size_t>(h0) * Nq : nullptr;
  return causal ? launch_fwd<128, true, 4, 0, 0, false, true>(mq, mk, mv, mo, oc, lc, nullptr, nullptr, nb, Nq, Nk, sl2,
                                                             1, st, rc, v_descale)
                : launch_fwd<128, false, 4, 0, 0, false, true>(mq, mk, mv, mo, oc, lc, nullptr, nullptr, nb, Nq, Nk, sl2,
                                                              1, st, rc, v_descale);
}

// The single-pass fp16 forward, once the arguments have been checked.
template <int EMU64 = kEmu64, int EMU128 = kEmu128>
int enqueue_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int Nq, int Nk, int D,
                float scale, int causal, cudaStream_t st, const RunCtl& rc) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, q, BH, Nq, D) || !make_map(&mk, k, BH, Nk, D) || !make_map(&mv, v, BH, Nk, D) ||
      !make_map(&mo, o, BH, Nq, D))
    return ATTN_ECUDA;
  const float sl2 = scale * 1.4426950408889634f;
  return dispatch_fwd<false, EMU64, EMU128>(D, causal, mq, mk, mv, mo, o, lse, nullptr, nullptr, BH, Nq, Nk, sl2, 1,
                                            st, rc);
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
             int D, float scale, int causal, void* stream) {
  bool empty = false;
  int rc = check_args(q, k, v, o, lse, B, H, Nq, Nk, D, scale, &empty);
  if (rc != ATTN_OK || empty) return rc;
  if ((rc = check_keys_per_pass(Nq, Nk, causal, 0)) != ATTN_OK) return rc;
  RunCtl run;
  if ((rc = enter(&run)) != ATTN_OK) return rc;
  return enqueue_fwd(q, k, v, o, lse, B * H, Nq, Nk, D, scale, causal, static_cast<cudaStream_t>(stream), run);
}

int attn_fwd_launch_count(int B, int H, int Nq, int Nk, int D, int causal) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 1 || (D != 64 && D != 128)) return -ATTN_EINVAL;
  if (B == 0 || H == 0 || Nq == 0) return 0;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ContextState* st = nullptr;
    const int r = context_state(&st);
    if (r != ATTN_OK) return -r;
    sms = st->sms;
  }
  const int64_t pairs = static_cast<int64_t>(B) * H * ((Nq + kRowsPerCta - 1) / kRowsPerCta);
  const int64_t q_tiles = static_cast<int64_t>(B) * H * ((Nq + kBlockM - 1) / kBlockM);
  const int64_t tail = tail_pairs(pairs, sms, (Nk + kBlockN - 1) / kBlockN, causal != 0, q_tiles);
  return (pairs - tail > 0 ? 1 : 0) + (tail > 0 ? 1 : 0);
}

size_t attn_splitkv_workspace_bytes(int B, int H, int Nq, int D, int num_splits) {
  if (B < 0 || H < 0 || Nq < 0 || (D != 64 && D != 128) || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_bytes(B, H, Nq, D, num_splits);
}

int attn_splitkv_suggest(int B, int H, int Nq, int Nk, int D, int causal) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (D != 64 && D != 128)) return 0;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ContextState* st = nullptr;
    if (context_state(&st) != ATTN_OK) return 0;
    sms = st->sms;
  }
  const int64_t ctas = static_cast<int64_t>(B) * H * ((Nq + kRowsPerCta - 1) / kRowsPerCta);
  const int64_t tiles = pair_key_tiles(Nq, Nk, causal);
  // No share may hold more keys than one pass may accumulate.
  const int64_t s_min = std::max<int64_t>(1, (tiles * kBlockN + ATTN_MAX_KEYS_PER_PASS - 1) / ATTN_MAX_KEYS_PER_PASS);
  // At least four key tiles per share, at most 256 shares.
  const int64_t s_max = std::max<int64_t>(s_min, std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, tiles / 4)));
  // Cost model in key-tile steps of one CTA (~1.1-1.4 us on GB300), fitted
  // to split-KV timings of decode and prefill shapes: waves of CTAs times
  // (the tiles of a share + ~5 steps of start-up and epilogue per CTA); a
  // split adds the merge launch (~8 steps) and the fp32 parts it writes and
  // reads back ((D+1)*4 bytes per row and share, both ways, at ~8 MB per
  // step).  One share means the single pass (no parts, no merge).
  const double rows = static_cast<double>(B) * H * Nq;
  int64_t best = s_min;
  double best_cost = 1e300;
  for (int64_t s = s_min; s <= s_max; ++s) {
    const double waves = static_cast<double>((ctas * s + sms - 1) / sms);
    double cost = waves * (static_cast<double>((tiles + s - 1) / s) + 5.0);
    if (s > 1) cost += 8.0 + rows * (D + 1) * 8.0 * static_cast<double>(s) / 8.0e6;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return static_cast<int>(std::min<int64_t>(best, kMaxSplits));
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                     int Nk, int D, float scale, int causal, int num_splits, void* workspace,
                     size_t workspace_bytes, void* stream) {
  bool empty = false;
  int rc = check_args(q, k, v, o, lse, B, H, Nq, Nk, D, scale, &empty);
  if (rc != ATTN_OK) return rc;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_EINVAL;
  if (empty) return ATTN_OK;
  const size_t need = splitkv_bytes(B, H, Nq, D, num_splits);
  if (!workspace || workspace_bytes < need) return ATTN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return ATTN_EUNSUPPORTED;
  const int BH = B * H;
  const size_t qbytes = static_cast<size_t>(BH) * Nq * D * 2, kvbytes = static_cast<size_t>(BH) * Nk * D * 2;
  if (ranges_overlap(workspace, need, q, qbytes) || ranges_overlap(workspace, need, k, kvbytes) ||
      ranges_overlap(workspace, need, v, kvbytes) || ranges_overlap(workspace, need, o, qbytes) ||
      (lse && ranges_overlap(workspace, need, lse, static_cast<size_t>(BH) * Nq * 4)))
    return ATTN_EUNSUPPORTED;
  if ((rc = check_keys_per_pass(Nq, Nk, causal, num_splits)) != ATTN_OK) return rc;
  RunCtl run;
  if ((rc = enter(&run)) != ATTN_OK) return rc;
  return enqueue_splitkv(q, k, v, o, lse, BH, Nq, Nk, D, scale, causal, num_splits, workspace,
                         static_cast<cudaStream_t>(stream), run);
}

int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                             int Nq, int Nk, int D, float scale, int causal, int num_splits, void* stream) {
  bool empty = false;
  int rc = check_args(q, k, v, o, lse, B, H, Nq, Nk, D, scale, &empty);
  if (rc != ATTN_OK) return rc;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_EINVAL;
  if (empty) return ATTN_OK;
  if (splitkv_bytes(B, H, Nq, D, num_splits) > kNoAllocScratchBytes) return ATTN_ESCRATCH;
  if ((rc = check_keys_per_pass(Nq, Nk, causal, num_splits)) != ATTN_OK) return rc;
  RunCtl run;
  if ((rc = enter(&run, true)) != ATTN_OK) return rc;
  return enqueue_splitkv(q, k, v, o, lse, B * H, Nq, Nk, D, scale, causal, num_splits, run.noalloc,
                         static_cast<cudaStream_t>(stream), run);
}

int attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                  void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int B, int H, int Nq, int Nk,
                  int D, float scale, int causal, int num_chunks, void* stream) {
  if (!q_host || !k_host || !v_host || !o_host) return ATTN_EINVAL;
  if ((lse_host == nullptr) != (lse_dev == nullptr)) return ATTN_EINVAL;
  if (num_chunks < 0 || num_chunks > kMaxHostChunks) return ATTN_EINVAL;
  bool empty = false;
  int rc = check_args(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, Nq, Nk, D, scale, &empty);
  if (rc != ATTN_OK || empty) return rc;
  const int BH = B * H;
  const size_t qb = static_cast<size_t>(BH) * Nq * D * 2, kb = static_cast<size_t>(BH) * Nk * D * 2;
  if (ranges_overlap(q_dev, qb, k_dev, kb) || ranges_overlap(q_dev, qb, v_dev, kb) ||
      ranges_overlap(k_dev, kb, v_dev, kb))
    return ATTN_EUNSUPPORTED;  // the device copies of the inputs are written here
  if ((rc = check_keys_per_pass(Nq, Nk, causal, 0)) != ATTN_OK) return rc;
  RunCtl run;
  if ((rc = enter(&run)) != ATTN_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ECUDA;
  const int chunks = std::max(1, std::min(num_chunks == 0 ? 32 : num_chunks, BH));
  auto compute = [&](int, int h0, int nb, cudaStream_t sc) -> int {
    const size_t qo = static_cast<size_t>(h0) * Nq * D, ko = static_cast<size_t>(h0) * Nk * D;
    return enqueue_fwd(static_cast<const __half*>(q_dev) + qo, static_cast<const __half*>(k_dev) + ko,
                       static_cast<const __half*>(v_dev) + ko, static_cast<__half*>(o_dev) + qo,
                       lse_dev ? lse_dev + static_cast<size_t>(h0) * Nq : nullptr, nb, Nq, Nk, D, scale, causal, sc,
                       run);
  };
  return host_pipeline(dev, q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev, BH, Nq,
                       Nk, D, 2, chunks, static_cast<cudaStream_t>(stream), compute);
}

size_t attn_fp8_workspace_bytes(int B, int H, int Nk, int D) {
  if (B < 0 || H < 0 || Nk < 0 || D != 128) return 0;
  return static_cast<size_t>(B) * H * D * ((static_cast<size_t>(Nk) + 15) / 16 * 16);
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                 int D, float scale, int causal, float q_descale, float k_descale, float v_descale, void* workspace,
                 size_t workspace_bytes, void* stream) {
  bool empty = false;
  int rc = check_args_fp8(q, k, v, o, lse, B, H, Nq, Nk, D, scale, q_descale, k_descale, v_descale, workspace,
                          workspace_bytes, &empty);
  if (rc != ATTN_OK || empty) return rc;
  RunCtl run;
  if ((rc = enter(&run)) != ATTN_OK) return rc;
  const float sl2 = scale * q_descale * k_descale * 1.4426950408889634f;
  return enqueue_fp8(q, k, v, o, lse, workspace, 0, B * H, Nq, Nk, sl2, v_descale, causal,
                     static_cast<cudaStream_t>(stream), run);
}

int attn_fwd_fp8_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                      void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int B, int H, int Nq,
                      int Nk, int D, float scale, int causal, float q_descale, float k_descale, float v_descale,
                      void* workspace, size_t workspace_bytes, int num_chunks, void* stream) {
  if (!q_host || !k_host || !v_host || !o_host) return ATTN_EINVAL;
  if ((lse_host == nullptr) != (lse_dev == nullptr)) return ATTN_EINVAL;
  if (num_chunks < 0 || num_chunks > kMaxHostChunks) return ATTN_EINVAL;
  bool empty = false;
  int rc = check_args_fp8(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, Nq, Nk, D, scale, q_descale, k_descale,
                          v_descale, workspace, workspace_bytes, &empty);
  if (rc != ATTN_OK || empty) return rc;
  const int BH = B * H;
  const size_t qb = static_cast<size_t>(BH) * Nq * D, kb = static_cast<size_t>(BH) * Nk * D;
  if (ranges_overlap(q_dev, qb, k_dev, kb) || ranges_overlap(q_dev, qb, v_dev, kb) ||
      ranges_overlap(k_dev, kb, v_dev, kb))
    return ATTN_EUNSUPPORTED;  // the device copies of the inputs are written here
  RunCtl run;
  if ((rc = enter(&run)) != ATTN_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ECUDA;
  const int chunks = std::max(1, std::min(num_chunks == 0 ? 32 : num_chunks, BH));
  const float sl2 = scale * q_descale * k_descale * 1.4426950408889634f;
  auto compute = [&](int, int h0, int nb, cudaStream_t sc) -> int {
    return enqueue_fp8(q_dev, k_dev, v_dev, o_dev, lse_dev, workspace, h0, nb, Nq, Nk, sl2, v_descale, causal, sc,
                       run);
  };
  return host_pipeline(dev, q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev, BH, Nq,
                       Nk, D, 1, chunks, static_cast<cudaStream_t>(stream), compute);
}

int attn_debug_pack_e4m3(const float* in, unsigned int* out, int n_quads, void* stream) {
  if (!in || !out || n_quads < 0) return ATTN_EINVAL;
  if (n_quads == 0) return ATTN_OK;
  attn_debug_pack_e4m3_kernel<<<(n_quads + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      in, reinterpret_cast<uint32_t*>(out), n_quads);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ECUDA;
}

int attn_debug_exp2_poly(const float* in, float* out, int n, void* stream) {
  if (n < 0) return ATTN_EINVAL;
  if (n == 0) return ATTN_OK;
  if (!in || !out) return ATTN_EINVAL;
  const int pairs = (n + 1) / 2;
  attn_debug_exp2_poly_kernel<<<(pairs + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ECUDA;
}

int attn_debug_fwd_poly_exp(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                            int Nk, int D, float scale, int causal, void* stream) {
  bool empty = false;
  int rc = check_args(q, k, v, o, lse, B, H, Nq, Nk, D, scale, &empty);
  if (rc != ATTN_OK || empty) return rc;
  if ((rc = check_keys_per_pass(Nq, Nk, causal, 0)) != ATTN_OK) return rc;
  RunCtl run;
  if ((rc = enter(&run)) != ATTN_OK) return rc;
  return enqueue_fwd<kDebugEmu, kDebugEmu>(q, k, v, o, lse, B * H, Nq, Nk, D, scale, causal,
                                           static_cast<cudaStream_t>(stream), run);
}

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument";
    case ATTN_EUNSUPPORTED: return "unsupported argument or device";
    case ATTN_ECUDA: return "CUDA error";
    case ATTN_ETIMEOUT: return "a kernel wait timed out";
    case ATTN_ESCRATCH: return "the problem needs more scratch than the library's built-in buffer holds";
    case ATTN_ETOOLONG: return "more keys per row in one pass than the accuracy limit allows: use attn_fwd_splitkv";
    default: return "unknown error code";
  }
}

int attn_get_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ECUDA;
  int h = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&h, g_attn_status, sizeof(int)) != cudaSuccess) return ATTN_ECUDA;
  if (h != 0 && cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess) return ATTN_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  ContextState* st = nullptr;
  if (context_state(&st) == ATTN_OK && st->status_host != nullptr) {
    volatile int* mirror = st->status_host;
    if (h == 0) h = *mirror;
    *mirror = 0;
  }
  return h;
}

int attn_debug_set(unsigned long long wait_timeout_ns, int drop_kv_tile) {
  if (wait_timeout_ns == 0 || drop_kv_tile < -1) return ATTN_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = wait_timeout_ns;
  g_drop_tile = drop_kv_tile;
  return ATTN_OK;
}

int attn_version(void) { return ATTN_VERSION; }

}  // extern "C"
