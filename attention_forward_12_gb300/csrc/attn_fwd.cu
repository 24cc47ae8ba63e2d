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
// sm_120; this one is built for the datacenter Blackwell tensor core:
//
//   * TMA producer (warp 4): loads the Q tile once and streams K and V tiles
//     through an NS-deep ring of 128B-swizzled shared-memory stages, each
//     stage guarded by full/empty mbarriers ("New Hardware: TMA": rank-N box
//     copies, hardware swizzle, one issuing thread, mbarrier transaction
//     counts; "Move 3 -- Pipelining": prefetch tile j+1 under tile j).
//   * MMA issuer (warp 5, one thread): S_j = Q K_j^T with tcgen05.mma
//     (A and B from shared memory) into one of two TMEM score buffers, and
//     O += P_j V_j with tcgen05.mma taking P from TMEM (the analogue of the
//     page's C->A register repack: P never goes through shared memory).
//     Double-buffered S lets S_{j+1} run on the tensor core while the
//     softmax warps work on S_j.
//   * Softmax warpgroup (warps 0-3, thread t owns query row t, which is
//     TMEM lane t): reads S_j with tcgen05.ld, masks, takes the row maximum,
//     computes p = 2^(s*scale*log2(e) - m) with the scale folded into one
//     FFMA, rounds p to fp16 and writes it back over S_j, sums it into d.
//     O is rescaled lazily: only when a row's maximum grows by more than
//     kTau (in log2 units) over the reference it was using; otherwise p is
//     taken against the stale reference, which is exact because p, d and o
//     share it (the conditional rescale the page credits to FlashAttention-4
//     in "Relationship to FA-3 and FA-4").  At the end it normalises O by d,
//     writes fp16 O and fp32 LSE.
//   * Causal (key j masked when j > i): a query tile visits only the key
//     tiles up to its diagonal, and only the diagonal and the ragged last
//     tile take the masked path.
//
// Every mbarrier wait is bounded (see WaitCtl): a wait that runs out raises
// the CTA's abort flag and the device status word, the CTA drains its TMA
// copies and tensor-core work in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "sm103_primitives.cuh"

using namespace attn_sm103;

namespace {

constexpr int kThreads = 192;   // 4 softmax warps + TMA warp + MMA warp
constexpr int kBlockM = 128;    // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;    // keys per tile
constexpr float kTau = 8.0f;    // lazy-rescale threshold, log2 units
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 64 fp16 (one swizzle column block)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

template <int HD, int NS>
struct Layout {
  static constexpr int kChunks = HD / 64;
  static constexpr uint32_t kTileBytes = kBlockM * HD * 2;  // Q, K or V tile
  static constexpr int kBars = 1 + 4 * NS + 2 + 2 + 1 + 1;
  static constexpr size_t kSmem = 1024 + kTileBytes * (1 + 2 * NS) + kBars * 8 + 8 + 8 + NS * 8;
};

}  // namespace

// Device status word: 0 = ok, otherwise the first ATTN_E* code a kernel
// recorded since the last attn_get_status().
__device__ int g_attn_status;

template <int HD, bool CAUSAL, int NS>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, __half* __restrict__ out,
                float* __restrict__ lse, int Nq, int Nk, float sl2, uint64_t timeout_ns,
                int drop_tile) {
  using L = Layout<HD, NS>;
  constexpr uint32_t TB = L::kTileBytes;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + TB;
  uint8_t* sV = sK + NS * TB;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(sV + NS * TB);
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;  // [2] S_j landed in TMEM buffer j&1
  uint64_t* p_full = s_full + 2;    // [2] P_j written over S_j (and O rescaled)
  uint64_t* o_done = p_full + 2;    // one phase per completed O += P V
  uint64_t* drain = o_done + 1;     // abort path only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* last_k = abort_flag + 1;     // [NS] last tile loaded per stage (abort drain)
  int* last_v = last_k + NS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int qt = CAUSAL ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  const int r0 = qt * kBlockM;
  const int kv_end = CAUSAL ? min(Nk, r0 + kBlockM) : Nk;
  const int nkv = (kv_end + kBlockN - 1) / kBlockN;  // >= 1

  // A CTA of a launch that already recorded an error does no work: after a
  // timeout the remaining CTAs exit at once instead of each waiting out its
  // own limit.  The status word is read by one thread and broadcast.
  if (threadIdx.x == 0) *abort_flag = *static_cast<volatile int*>(&g_attn_status);
  __syncthreads();
  if (*abort_flag) return;

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
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], kBlockM);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem;        // columns [0,128): S / P buffer 0
  const uint32_t tS1 = tmem + 128;  // columns [128,256): S / P buffer 1
  const uint32_t tO = tmem + 256;   // columns [256, 256+HD): O accumulator
  const WaitCtl wc{abort_flag, &g_attn_status, timeout_ns};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      mbar_arrive_expect_tx(q_full, TB);
      for (int c = 0; c < L::kChunks; ++c) tma_load_3d(sQ + c * kChunkBytes, &tmQ, q_full, c * 64, r0, bh);
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (j >= NS) ok = mbar_wait(&k_empty[s], ph ^ 1, wc, ATTN_ETIMEOUT);
        if (!ok) break;
        if (j != drop_tile) {  // drop_tile >= 0 only under attn_debug_set
          mbar_arrive_expect_tx(&k_full[s], TB);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sK + s * TB + c * kChunkBytes, &tmK, &k_full[s], c * 64, j * kBlockN, bh);
          last_k[s] = j;
        }
        if (j >= NS) ok = mbar_wait(&v_empty[s], ph ^ 1, wc, ATTN_ETIMEOUT);
        if (!ok) break;
        mbar_arrive_expect_tx(&v_full[s], TB);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sV + s * TB + c * kChunkBytes, &tmV, &v_full[s], c * 64, j * kBlockN, bh);
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
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f16_f32(kBlockM, kBlockN, false, false);
      constexpr uint32_t kIdescPV = idesc_f16_f32(kBlockM, HD, false, true);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(q_full, 0, wc, ATTN_ETIMEOUT);
      if (ok) tc_fence_after();
      for (int j = 0; j <= nkv && ok; ++j) {
        if (j < nkv) {
          // S_j = Q K_j^T : both operands K-major, 128B swizzle; K = HD in
          // steps of 16 (32 bytes inside a 128-byte swizzle row).
          const int s = j % NS;
          ok = mbar_wait(&k_full[s], (j / NS) & 1, wc, ATTN_ETIMEOUT);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dS = (j & 1) ? tS1 : tS0;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            umma_ss(dS, smem_desc(aQ + off, 16, 1024), smem_desc(aK + s * TB + off, 16, 1024), kIdescQK,
                    kk > 0 ? 1u : 0u);
          }
          umma_commit(&k_empty[s]);
          umma_commit(&s_full[j & 1]);
        }
        if (j >= 1) {
          // O += P_t V_t : P (fp16, packed two per column) from TMEM as the
          // A operand, V from shared memory MN-major (rows = keys, 128 bytes
          // of D per row; LBO = next 64 columns of D, SBO = next 8 keys).
          const int t = j - 1;
          const int s = t % NS;
          ok = mbar_wait(&p_full[t & 1], (t >> 1) & 1, wc, ATTN_ETIMEOUT);
          if (ok) ok = mbar_wait(&v_full[s], (t / NS) & 1, wc, ATTN_ETIMEOUT);
          if (!ok) break;
          tc_fence_after();
          const uint32_t aP = (t & 1) ? tS1 : tS0;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            umma_ts(tO, aP + kk * 8, smem_desc(aV + s * TB + kk * 2048, kChunkBytes, 1024), kIdescPV,
                    (t > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&v_empty[s]);
          umma_commit(o_done);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // tile row == TMEM lane
    const int i = r0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int row_lim = CAUSAL ? min(Nk, i + 1) : Nk;  // admissible keys: [0, row_lim)
    float m_ref = -INFINITY;  // reference maximum, log2 units of the scaled score
    float dsum = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const uint32_t tS = (j & 1) ? tS1 : tS0;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, wc, ATTN_ETIMEOUT));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);

      const int key0 = j * kBlockN;
      const bool masked = (key0 + kBlockN > Nk) || (CAUSAL && key0 + kBlockN - 1 > r0);
      const int lim = row_lim - key0;  // columns [0, lim) of this tile are admissible
      float mx = -INFINITY;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const bool valid = (c * 32 + e) < lim;
            const float x = valid ? __uint_as_float(sr[c][e]) : -INFINITY;
            sr[c][e] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sr[c][e]));
      }
      const float mt = (mx == -INFINITY) ? -INFINITY : mx * sl2;
      const bool resc = mt > m_ref + kTau;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_ref - mt);  // 0 on the first tile (m_ref = -inf)
        m_ref = mt;
        dsum *= alpha;
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;

      // p = 2^(s*sl2 - m_ref), rounded to fp16 precision in fp32 so that the
      // denominator sums exactly the weights the tensor core multiplies V by.
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][e]), sl2, neg_m));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[c][e + 1]), sl2, neg_m));
          if (masked) {
            p0 = (c * 32 + e) < lim ? p0 : 0.f;
            p1 = (c * 32 + e + 1) < lim ? p1 : 0.f;
          }
          p0 = __uint_as_float((__float_as_uint(p0) + 0x1000u) & 0xFFFFE000u);
          p1 = __uint_as_float((__float_as_uint(p1) + 0x1000u) & 0xFFFFE000u);
          rs0 += p0;
          rs1 += p1;
          const __half2 h2 = __floats2half2_rn(p0, p1);
          pk[c >> 1][(c & 1) * 16 + (e >> 1)] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      dsum += rs0 + rs1;
      tmem_st32(tS + lane_off, pk[0]);
      tmem_st32(tS + lane_off + 32, pk[1]);

      if (j >= 1) {
        // O must hold exactly P_0..P_{j-1} before it is rescaled and before
        // P_j is released; every completion of O += P V is observed in order.
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, wc, ATTN_ETIMEOUT));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32(tO + lane_off + c * 32, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32(tO + lane_off + c * 32, orr);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (nkv - 1) & 1, wc, ATTN_ETIMEOUT));
    if (ok) {
      // ---------------------------------------------------------- epilogue
      tc_fence_after();
      const float inv = 1.f / dsum;
      __half* orow = out + (static_cast<size_t>(bh) * Nq + i) * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(tO + lane_off + c * 32, orr);
        tmem_ld_wait(orr);
        if (i < Nq) {
          uint32_t h[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __half2 h2 = __floats2half2_rn(__uint_as_float(orr[2 * e]) * inv,
                                                 __uint_as_float(orr[2 * e + 1]) * inv);
            h[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(h[4 * e], h[4 * e + 1], h[4 * e + 2], h[4 * e + 3]);
        }
      }
      if (lse != nullptr && i < Nq) lse[static_cast<size_t>(bh) * Nq + i] = (m_ref + log2f(dsum)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out somewhere in this CTA: let every TMA copy and every
    // tensor-core op it issued land before the shared memory and TMEM go.
    if (warp == 4 && lane == 0) {
      mbar_wait(q_full, 0, wc, ATTN_ETIMEOUT, false);
      for (int s = 0; s < NS; ++s) {
        if (last_k[s] >= 0) mbar_wait(&k_full[s], (last_k[s] / NS) & 1, wc, ATTN_ETIMEOUT, false);
        if (last_v[s] >= 0) mbar_wait(&v_full[s], (last_v[s] / NS) & 1, wc, ATTN_ETIMEOUT, false);
      }
    }
    if (warp == 5 && lane == 0) {
      umma_commit(drain);
      mbar_wait(drain, 0, wc, ATTN_ETIMEOUT, false);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// =====================================================================
// Host side
// =====================================================================
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
uint64_t g_timeout_ns = kDefaultTimeoutNs;
int g_drop_tile = -1;
constexpr int kMaxDevices = 64;
int g_dev_ready[kMaxDevices];  // 1 = attributes set and device checked; -1 = unsupported

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
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

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

template <int HD, bool CAUSAL, int NS>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* o, float* lse, int BH,
           int Nq, int Nk, float sl2, cudaStream_t st, uint64_t timeout_ns, int drop) {
  using L = Layout<HD, NS>;
  auto kern = attn_fwd_kernel<HD, CAUSAL, NS>;
  static_assert(L::kSmem <= 232448, "shared memory budget");
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kSmem)) !=
      cudaSuccess)
    return ATTN_ECUDA;
  dim3 grid((Nq + kBlockM - 1) / kBlockM, BH, 1);
  kern<<<grid, kThreads, L::kSmem, st>>>(mq, mk, mv, static_cast<__half*>(o), lse, Nq, Nk, sl2, timeout_ns, drop);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ECUDA;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
             int D, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o) return ATTN_EINVAL;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 1) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_EINVAL;
  if (D != 64 && D != 128) return ATTN_EUNSUPPORTED;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_EUNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 65535) return ATTN_EUNSUPPORTED;
  if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;  // empty output: nothing to do
  const int BH = B * H;
  const size_t qbytes = static_cast<size_t>(BH) * Nq * D * 2, kvbytes = static_cast<size_t>(BH) * Nk * D * 2;
  if (ranges_overlap(o, qbytes, q, qbytes) || ranges_overlap(o, qbytes, k, kvbytes) ||
      ranges_overlap(o, qbytes, v, kvbytes))
    return ATTN_EUNSUPPORTED;
  if (lse && (ranges_overlap(lse, static_cast<size_t>(BH) * Nq * 4, o, qbytes) ||
              ranges_overlap(lse, static_cast<size_t>(BH) * Nq * 4, q, qbytes) ||
              ranges_overlap(lse, static_cast<size_t>(BH) * Nq * 4, k, kvbytes) ||
              ranges_overlap(lse, static_cast<size_t>(BH) * Nq * 4, v, kvbytes)))
    return ATTN_EUNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ECUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev_ready[dev] == 0) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_ECUDA;
      g_dev_ready[dev] = (prop.major == 10 && prop.minor == 3) ? 1 : -1;
    }
    if (g_dev_ready[dev] < 0) return ATTN_EUNSUPPORTED;
  }
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, BH, Nq, D) || !make_map(&mk, k, BH, Nk, D) || !make_map(&mv, v, BH, Nk, D))
    return ATTN_ECUDA;
  uint64_t timeout;
  int drop;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    timeout = g_timeout_ns;
    drop = g_drop_tile;
  }
  const float sl2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (D == 64)
    return causal ? launch<64, true, 4>(mq, mk, mv, o, lse, BH, Nq, Nk, sl2, st, timeout, drop)
                  : launch<64, false, 4>(mq, mk, mv, o, lse, BH, Nq, Nk, sl2, st, timeout, drop);
  return causal ? launch<128, true, 2>(mq, mk, mv, o, lse, BH, Nq, Nk, sl2, st, timeout, drop)
                : launch<128, false, 2>(mq, mk, mv, o, lse, BH, Nq, Nk, sl2, st, timeout, drop);
}

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument";
    case ATTN_EUNSUPPORTED: return "unsupported argument or device";
    case ATTN_ECUDA: return "CUDA error";
    case ATTN_ETIMEOUT: return "a kernel wait timed out";
    default: return "unknown error code";
  }
}

int attn_get_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ECUDA;
  int h = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&h, g_attn_status, sizeof(int)) != cudaSuccess) return ATTN_ECUDA;
  if (h != 0 && cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess) return ATTN_ECUDA;
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
