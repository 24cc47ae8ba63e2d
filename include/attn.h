/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * The operation is the one the pages build up in "Learning FlashAttention
 * the Hard Way -- Part 2" (problem statement: F.scaled_dot_product_attention
 * on fp16 [B,H,N,D] tensors, the SDPA_P / SDPA_L shapes; the streaming
 * (m, d, o) reduction of sections "Move 0" and "Move 1 -- Tensor Cores"):
 *
 *     O[b,h,i,:] = sum_j softmax_j(scale * q[b,h,i,:] . k[b,h,j,:]) v[b,h,j,:]
 *     LSE[b,h,i] = log sum_j exp(scale * q[b,h,i,:] . k[b,h,j,:])   (natural log)
 *
 * over the admissible keys j: all 0 <= j < Nk, or, when causal, only j <= i
 * (top-left alignment: key j is masked when j > i, as torch's is_causal).
 * The N x N scores never reach global memory.
 *
 * Conventions shared by every entry point:
 *   - Pointers to tensors are DEVICE pointers on the current CUDA device.
 *     The caller owns every buffer; the library allocates nothing per call.
 *   - Layout is contiguous row-major: q and o are [B,H,Nq,D], k and v are
 *     [B,H,Nk,D], lse is [B,H,Nq]; element (b,h,n,d) of q is at
 *     ((b*H + h)*Nq + n)*D + d.
 *   - q, k, v, o are IEEE binary16 (fp16); lse is fp32.  Products are
 *     accumulated in fp32; the softmax weights are rounded to fp16 before
 *     they multiply V (as the page's C->A repack rounds P with cvt.rn).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on that stream; they perform no host synchronisation
 *     and no allocation, so they can be captured in a CUDA graph (make one
 *     ordinary call on the device first: it sets the kernels' attributes and
 *     creates the host copy of the device's status word, see attn_fwd).
 *   - Return values are ATTN_* codes below.  Argument errors are detected on
 *     the host before anything is enqueued.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_VERSION 4

enum {
  ATTN_OK = 0,
  ATTN_EINVAL = 1,        /* null tensor pointer, negative size, Nk < 1, scale < 0 or not finite */
  ATTN_EUNSUPPORTED = 2,  /* D not in {64,128}, misaligned pointer, overlapping output,
                             B*H > 65535, or a device other than sm_103 */
  ATTN_ECUDA = 3,         /* tensor-map encoding or kernel launch failed */
  ATTN_ETIMEOUT = 4,      /* a kernel wait ran out: reported by attn_get_status, and by every
                             call made while that report is pending */
  ATTN_ESCRATCH = 5,      /* attn_fwd_splitkv_noalloc: problem larger than the built-in scratch */
  ATTN_ETOOLONG = 6       /* more keys per row in one pass than ATTN_MAX_KEYS_PER_PASS: use
                             attn_fwd_splitkv with more shares */
};

/* The most keys one row may accumulate in a single pass of the fp16 forward
 * (2^19).  O is summed in fp32 by the tensor core over every key tile of the
 * pass, and that sum drifts with the number of tiles: measured against an
 * fp64 reference on N(0,1) data, the relative RMS error of O is 2.8e-4 at
 * 2^16 keys, 5.8e-4 at 2^19 and 1.1e-3 at 2^20, past the 1e-3 this library
 * is held to.  Longer rows go through attn_fwd_splitkv, whose shares are
 * summed separately and merged in fp32 (2.1e-4 at 2^20 with 16 shares). */
#define ATTN_MAX_KEYS_PER_PASS 524288

/* Size of the device buffer compiled into the library for
 * attn_fwd_splitkv_noalloc (64 MiB on every device that loads the library). */
#define ATTN_NOALLOC_SCRATCH_BYTES (64ull * 1024ull * 1024ull)

/*
 * attn_fwd -- O = softmax(scale * Q K^T) V and LSE, fp16 in/out.
 *
 *   q      [B,H,Nq,D] fp16, 16-byte aligned.
 *   k, v   [B,H,Nk,D] fp16, 16-byte aligned.
 *   o      [B,H,Nq,D] fp16, 16-byte aligned, written; must not overlap q, k, v.
 *   lse    [B,H,Nq] fp32, 4-byte aligned, written; may be NULL (not computed).
 *   B, H, Nq >= 0 (any of them 0: nothing is done, ATTN_OK), Nk >= 1,
 *   B*H <= 65535, D in {64, 128}.
 *   scale  softmax scale, finite and >= 0 (the pages use 1/sqrt(D)).
 *   causal 0: every key is admissible; nonzero: key j masked when j > i.
 *
 * Enqueues one kernel on `stream`, or two for the non-causal forward when
 * the last wave of CTAs would occupy at most half the SMs
 * (attn_fwd_launch_count tells which); the second is a programmatic
 * dependent launch of the first, and the call as a whole completes in
 * stream order.  The kernels allow programmatic dependents to start early:
 * a kernel the caller launches next with programmatic stream serialization
 * must wait on its grid dependency (cudaGridDependencySynchronize) before it
 * reads O or LSE, as that feature requires anyway.
 *
 * Key range: the keys one row accumulates -- Nk, or min(Nk, Nq) when causal
 * -- must not exceed ATTN_MAX_KEYS_PER_PASS (2^19), else ATTN_ETOOLONG is
 * returned and nothing is enqueued; attn_fwd_splitkv takes longer rows.
 *
 * Errors: ATTN_EINVAL / ATTN_EUNSUPPORTED / ATTN_ETOOLONG for bad arguments
 * (nothing is enqueued), ATTN_ECUDA if encoding the TMA descriptors or the
 * launch fails.  A kernel whose internal wait runs out stops early, leaves
 * o / lse undefined and records ATTN_ETIMEOUT in the device's status word,
 * of which the library keeps a copy in page-locked host memory.  From the
 * moment that copy shows the error until attn_get_status() reads and clears
 * it, every forward entry point returns ATTN_ETIMEOUT at once, without
 * enqueueing anything and without synchronising; launches that were already
 * enqueued when the error was recorded do no work (their outputs are
 * undefined).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
             int Nk, int D, float scale, int causal, void* stream);

/*
 * The number of kernels attn_fwd enqueues for these sizes on the current
 * device: 1, or 2 for the non-causal forward when the query-tile pairs of a
 * last partial wave that would occupy at most half the SMs run as a second
 * launch of single-query-tile CTAs after full waves of pairs (done when a
 * query tile has 16 key tiles or more; a grid of less than half a wave,
 * a causal grid of at most one wave, or a grid of half-empty pairs that
 * takes clearly fewer waves that way, runs as single-query-tile CTAs
 * alone, in one launch).  0
 * when there is nothing to compute.  For counting launches, e.g. in a
 * benchmark.  Returns
 * -ATTN_EINVAL for bad sizes, -ATTN_EUNSUPPORTED / -ATTN_ECUDA when the
 * current device cannot be used.
 */
int attn_fwd_launch_count(int B, int H, int Nq, int Nk, int D, int causal);

/*
 * attn_fwd_host -- attn_fwd for tensors in HOST memory: copies Q, K and V
 * to the caller's device buffers, runs the forward and copies O and LSE back,
 * with the three overlapped.  The heads (the flattened B*H) are cut into
 * num_chunks contiguous groups; chunk c's host-to-device copy, its forward
 * and its device-to-host copy run on internal streams (one for the copies
 * in, two for the forwards, taken in turn so that consecutive chunks share
 * the SMs at their boundary, one for the copies out), so chunk c+1 is copied
 * in while chunk c is computed and chunk c-1 copied out.  (The
 * pages have no counterpart: this is the library's end-to-end entry point.)
 *
 *   q_host, k_host, v_host, o_host, lse_host  host tensors, same layouts as
 *          attn_fwd.  Page-locked (pinned) memory is needed for the copies
 *          to overlap; pageable memory works, slower.  lse_host may be NULL
 *          (then lse_dev must be NULL too).
 *   q_dev, k_dev, v_dev, o_dev, lse_dev  device buffers of the full sizes,
 *          with attn_fwd's alignment and overlap rules (q/k/v also must not
 *          overlap one another); the inputs are copied into them and the
 *          outputs computed there, so they hold the same data as after
 *          attn_fwd when the call completes.
 *   num_chunks  1 .. 64, or 0 for the default (32); capped at B*H.
 *   B, H, Nq, Nk, D, scale, causal: as attn_fwd.
 *   stream  the work starts after everything already queued on `stream`
 *          and `stream` waits for the last output copy: synchronise it
 *          before reading o_host / lse_host.
 *
 * The internal streams and events are created once per device, on the
 * first call (make that call before any stream capture), and reused; calls
 * from several host threads serialise on them.  Nothing is allocated per
 * call.  Errors: as attn_fwd, plus ATTN_EINVAL for a null host tensor,
 * lse_host and lse_dev not both given or both NULL, or num_chunks outside
 * 0..64.
 */
int attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                  void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int B, int H, int Nq,
                  int Nk, int D, float scale, int causal, int num_chunks, void* stream);

/*
 * attn_fwd_splitkv -- the same forward, with the keys of every query tile
 * divided into num_splits contiguous shares that separate CTAs compute in
 * parallel, followed by a merge.  This is the split-KV / Flash-Decoding
 * form the page names in "Relationship to FA-3 and FA-4" ("the monoid's
 * split-K"): each share yields a partial carrier (its normalised output and
 * log-sum-exp), and a second kernel combines the shares with the carrier
 * merge  (m1,d1,o1) (+) (m2,d2,o2) = (m, d1 e^(m1-m) + d2 e^(m2-m),
 * o1 e^(m1-m) + o2 e^(m2-m)),  m = max(m1, m2).  It pays off when
 * B*H*ceil(Nq/256) is small next to the SM count (decoding against a long key
 * sequence); results equal attn_fwd's within rounding.
 *
 *   q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, stream: as attn_fwd.
 *   num_splits  1 .. 256 shares (attn_splitkv_suggest gives one); shares
 *               that hold no admissible key are allowed.  A share holds
 *               ceil(T / num_splits) key tiles of 128 at most, T being the
 *               key tiles of the longest query-tile pair (ceil(Nk / 128); when
 *               causal, ceil(min(Nk, Nq rounded up to 256) / 128)); that times
 *               128 must not exceed ATTN_MAX_KEYS_PER_PASS, else
 *               ATTN_ETOOLONG.
 *   workspace   device memory owned by the caller, 16-byte aligned, at least
 *               attn_splitkv_workspace_bytes(B, H, Nq, D, num_splits) bytes,
 *               not overlapping any tensor argument.  Its contents on entry
 *               do not matter; it is overwritten.  Two calls that use the
 *               same workspace must not run concurrently on the GPU.
 *
 * Enqueues two kernels on `stream`.  Errors as attn_fwd, plus ATTN_EINVAL for
 * num_splits outside 1..256 or a missing / too small workspace and
 * ATTN_EUNSUPPORTED for a misaligned or overlapping workspace.  The merge
 * kernel, too, does nothing while the device's status word holds an error.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int Nq, int Nk, int D, float scale, int causal, int num_splits, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Bytes of workspace attn_fwd_splitkv needs: num_splits*B*H*Nq*(D+1)*4.
 * 0 for negative sizes, D not in {64,128} or num_splits outside 1..256. */
size_t attn_splitkv_workspace_bytes(int B, int H, int Nq, int D, int num_splits);

/* A share count for the current device, from a cost model of the kernels
 * measured on GB300: waves of CTAs times the key tiles of a share plus a
 * fixed cost per CTA, and for a split the merge and the fp32 parts written
 * and read back.  1 means the single pass (attn_fwd) is expected to be
 * faster: a grid that already fills the SMs gains nothing from shares.
 * Shares hold at least four 128-key tiles and at most
 * ATTN_MAX_KEYS_PER_PASS keys.  Returns >= 1, or 0 for bad arguments or
 * when the current device is not supported. */
int attn_splitkv_suggest(int B, int H, int Nq, int Nk, int D, int causal);

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv for callers that cannot
 * allocate device memory.  Some callers are not allowed to call cudaMalloc
 * or to hand out a workspace: a serving loop that must never enter an
 * allocator once it is running (allocation can stall or fail under memory
 * pressure), or a plugin whose host framework owns all device memory and
 * passes in only the tensors.  This entry point takes no workspace; the
 * shares' partial results go to a fixed scratch buffer built into the
 * library instead.  (The pages have no counterpart: this is a packaging
 * choice of this library, not part of the method.)
 *
 *   Arguments and results: as attn_fwd_splitkv, without workspace arguments.
 *   Limit: the problem must fit the buffer,
 *     num_splits * B * H * Nq * (D + 1) * 4 <= ATTN_NOALLOC_SCRATCH_BYTES,
 *   else ATTN_ESCRATCH is returned and nothing is enqueued.
 *   The buffer is held by every device that loads the library, until the
 *   process exits.  Every call looks up the buffer's device address with
 *   cudaGetSymbolAddress (a runtime query that allocates nothing), so the
 *   address stays right after a context reset.  The first call on a device
 *   loads the library's kernels there; make that first call before any
 *   stream capture.
 *   Every call uses the same buffer, which keeps the last call's contents;
 *   nothing in it needs to start at zero (each part is written before it
 *   is read).  Calls whose kernels overlap on the GPU race on the buffer:
 *   order them (one stream, or events between streams).
 *   The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *   library routine.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                             int Nq, int Nk, int D, float scale, int causal, int num_splits, void* stream);

/*
 * attn_fwd_fp8 -- the forward on 8-bit inputs: Q, K and V in OCP FP8 E4M3
 * (one byte each; 4 exponent bits, bias 7, 3 mantissa bits, largest finite
 * value 448), both products on the tensor core's 8-bit path with fp32
 * accumulation.  This is the lower-precision route the pages point to for
 * the newer tensor cores ("faster lower-precision tensor cores"; FA-3 and
 * FA-4's low-precision paths in "Relationship to FA-3 and FA-4"); the pages
 * give no kernel for it, and this one is the fp16 kernel with 8-bit
 * operands:
 *
 *   S = scale * (q_descale Q)(k_descale K)^T,  p = 2^(S log2 e - m),
 *   P rounded to E4M3 (round to nearest even; p <= 256 by the lazy rescale,
 *   inside the format's range), O = v_descale * (P V) / sum p  in fp16,
 *   LSE as attn_fwd, of the descaled scores.
 *
 *   q      [B,H,Nq,128] E4M3 bytes, 16-byte aligned.
 *   k, v   [B,H,Nk,128] E4M3 bytes, 16-byte aligned.
 *   o      [B,H,Nq,128] fp16, 16-byte aligned, written; lse as attn_fwd.
 *   q_descale, k_descale, v_descale  per-tensor factors, finite and > 0,
 *          that the stored values are multiplied by (1 for unscaled data).
 *   workspace  device memory owned by the caller, 16-byte aligned, at least
 *          attn_fp8_workspace_bytes(B, H, Nk, D) bytes, not overlapping any
 *          tensor: receives V transposed ([B,H,128,Nk] with rows rounded up
 *          to 16 bytes), which the P V product reads with keys contiguous.
 *          Two calls that share a workspace must not run concurrently.
 *   B, H, Nq, Nk, scale, causal, stream: as attn_fwd.  D must be 128.
 *
 * Enqueues the transpose, then the forward's kernels, on `stream`: one
 * more than attn_fwd_launch_count(B, H, Nq, Nk, 128, causal), the forward
 * following the same rule as attn_fwd's on when its last partial wave runs
 * as a second launch of single-query-tile CTAs.
 * Errors as attn_fwd, plus ATTN_EINVAL for a descale that is not finite and
 * positive or a missing / too small workspace, ATTN_EUNSUPPORTED for D != 128
 * or a misaligned or overlapping workspace.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                 int Nk, int D, float scale, int causal, float q_descale, float k_descale, float v_descale,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_fp8_host -- attn_fwd_fp8 for tensors in HOST memory, pipelined
 * over chunks of heads like attn_fwd_host (copies in, V transpose and
 * forward, copies out, overlapped).  Host tensors: q_host, k_host, v_host in
 * E4M3, o_host fp16, lse_host fp32 (may be NULL, then lse_dev too); device
 * buffers of the full sizes and the workspace with attn_fwd_fp8's rules;
 * num_chunks and stream as attn_fwd_host.  Errors as attn_fwd_fp8 and
 * attn_fwd_host.
 */
int attn_fwd_fp8_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                      void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int B, int H, int Nq,
                      int Nk, int D, float scale, int causal, float q_descale, float k_descale, float v_descale,
                      void* workspace, size_t workspace_bytes, int num_chunks, void* stream);

/* Bytes of workspace attn_fwd_fp8 needs: B*H*D*round_up(Nk, 16).  0 for
 * negative sizes or D != 128. */
size_t attn_fp8_workspace_bytes(int B, int H, int Nk, int D);

/*
 * Testing hook: the E4M3 rounding the FP8 forward applies to P, on its own.
 * in: 4*n_quads fp32 values (device); out: n_quads words (device), word i
 * holding in[4i] in bits 0-7 ... in[4i+3] in bits 24-31.  Asynchronous on
 * `stream`.  ATTN_EINVAL for null pointers or n_quads < 0.
 */
int attn_debug_pack_e4m3(const float* in, unsigned int* out, int n_quads, void* stream);

/*
 * Testing hook: the FMA-pipe 2^x of the forward ("the FMA-emulated exp" of
 * FlashAttention-4 in "Relationship to FA-3 and FA-4": Cody-Waite reduction
 * to [-1/2, 1/2], a degree-4 minimax polynomial, the exponent added to the
 * float's exponent field), on its own.  in, out: n fp32 values (device);
 * out[i] = 2^in[i] with relative error below 4e-6 for -126 <= in[i] <= 127;
 * inputs below -126, and NaN, give 2^-126.  Asynchronous on `stream`.
 * n = 0 does nothing (the pointers may then be NULL); ATTN_EINVAL for null
 * pointers with n > 0, or n < 0.
 */
int attn_debug_exp2_poly(const float* in, float* out, int n, void* stream);

/*
 * Testing hook: attn_fwd with one pair of exponentials in four taken by the
 * FMA-pipe polynomial above instead of the exponential unit (the forward
 * itself uses the exponential unit alone: on GB300 the split measured
 * slower).  Arguments, results and errors as attn_fwd.
 */
int attn_debug_fwd_poly_exp(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int Nq, int Nk, int D, float scale, int causal, void* stream);

/* Human-readable text for an ATTN_* code.  Never NULL. */
const char* attn_strerror(int code);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word and its host copy: ATTN_OK, or the first error a kernel recorded
 * since the last call (ATTN_ETIMEOUT).  Returns ATTN_ECUDA if the
 * synchronisation itself fails.
 */
int attn_get_status(void* stream);

/*
 * Testing hook.  Sets the limit of every kernel wait (nanoseconds of GPU
 * global time, default 2e9) and, when drop_kv_tile >= 0, makes the producer
 * skip the K load of that key tile so that the wait for it runs out; -1
 * restores normal operation.  Affects calls made after it, process-wide.
 * Returns ATTN_EINVAL for a zero timeout or drop_kv_tile < -1.
 */
int attn_debug_set(unsigned long long wait_timeout_ns, int drop_kv_tile);

/* ATTN_VERSION of the library. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
