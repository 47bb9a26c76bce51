/*
 * flamia.h - C ABI of the GB300 (sm_103a) MXFP8 causal packed attention library.
 *
 * The method is the MXFP8 training path of "FLAMIA: FLAsh MIcroscaling
 * Attention for Fast and Causally Safe Training on Blackwell" (arXiv
 * 2611.03344): softmax attention over documents packed into one token
 * sequence, with E4M3 operands carrying one UE8M0 (power-of-two) scale per
 * 32 contraction elements, forward and backward.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument named *_dev is a CUDA device pointer owned by the
 *    caller.  The library never allocates, frees or synchronizes inside these
 *    calls; each call only enqueues kernels on `stream` (a cudaStream_t passed
 *    as void*, NULL = legacy default stream) of the current device.
 *  - Packed layout (the "varlen" convention): token t of the packed sequence,
 *    head h, channel c of a [T, H, d] tensor sits at ((t * H) + h) * d + c.
 *    bf16 tensors are IEEE bfloat16 stored as uint16.
 *  - cu_seqlens_dev: int32 [n_docs + 1], non-decreasing, cu[0] >= 0,
 *    cu[n_docs] <= T.  Document r is tokens [cu[r], cu[r+1]); empty documents
 *    are allowed.  Tokens before cu[0] or at/after cu[n_docs] belong to no
 *    document: their outputs are O = 0, LSE = +inf, dQ = dK = dV = 0.
 *    The table is read on the device only; a malformed table is detected
 *    there, reported through flamia_get_status(), and the attention kernels
 *    then do no work.
 *  - d must be 64 or 128; Hq % Hkv == 0 (grouped-query heads: query head h
 *    reads key/value head h / (Hq / Hkv)); T >= 1; T * max(Hq, Hkv) * d
 *    < 2^31; all pointers 16-byte aligned.
 *  - Return value: 0 = enqueued; a negative FLAMIA_ERR_* code = rejected on the
 *    host before any launch (nothing was enqueued).
 *  - Scale tables ("*_scales") hold one UE8M0 byte per (head, token), layout
 *    [H, T]: byte = E + 127 for the power-of-two scale 2^E of the token's
 *    32-token block.  Codes ("*_codes") are E4M3 bytes in the packed layout.
 */
#ifndef FLAMIA_H_
#define FLAMIA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FLAMIA_OK 0
#define FLAMIA_ERR_ARG -1           /* null pointer, bad size, Hq % Hkv != 0, bad c/tau */
#define FLAMIA_ERR_UNSUPPORTED_D -2 /* d not in {64, 128} */
#define FLAMIA_ERR_ALIGN -3         /* a pointer is not 16-byte aligned */
#define FLAMIA_ERR_LAUNCH -4        /* a CUDA launch or tensor-map encode failed */
#define FLAMIA_ERR_DEVICE -5        /* the current device is not a Blackwell (sm_10x) GPU */
#define FLAMIA_ERR_NOALLOC_LIMIT -6 /* problem larger than flamia_fwd_noalloc's fixed scratch allows */
#define FLAMIA_ERR_UNSUPPORTED_OPT -7 /* an option combination this call does not implement (exact, nvfp4 or deterministic_dq while the score-tile dump is set) */

/* Device status word values (flamia_get_status). */
#define FLAMIA_STATUS_OK 0
#define FLAMIA_STATUS_BAD_SEQLENS 1 /* cu_seqlens not monotone or beyond T */
#define FLAMIA_STATUS_TIMEOUT 2     /* an on-chip wait exceeded its time budget */

typedef struct flamia_opts {
  /* Fixed multiplier 2^c_exp applied to probabilities before their E4M3
   * rounding, and the conditional-rescale threshold tau (log2 units): a
   * query row's running maximum is only replaced when a key tile raises it
   * by more than tau.  Must satisfy c_exp + tau <= log2(448) ~ 8.8 (FLAMIA
   * Section 3.4 and Appendix B.1: beyond it probabilities saturate silently);
   * the call is rejected otherwise.  MXFP8 uses c = 4, tau = 4. */
  int32_t c_exp;
  int32_t tau;
  /* 1 = causal (key j visible to query i iff j <= i within the document),
   * 0 = every key of the document is visible. */
  int32_t causal;
  /* 1 = rotate Q and K along the head dimension with the Sylvester Hadamard
   * matrix H_d before they are quantized (FLAMIA Section 3.4 and Appendix
   * A.2: the shared orthogonal transform leaves Q K^T unchanged and spreads
   * channel outliers).  The rotation is computed in fp32 by radix-2
   * butterflies (strides 1, 2, ..., d/2, lower element first); scores take
   * the factor 1/d out, and flamia_bwd maps dQ and dK back with H_d / d, so
   * the same value must be passed to both calls.  d = 128 only (rejected
   * with FLAMIA_ERR_ARG otherwise).  0 = no rotation (the default). */
  int32_t hadamard;
  /* 1 = the exact options of FLAMIA Section 3.2 and Appendix A.3.  Q, K, V
   * (and in flamia_bwd dO) get one exponent per token and head instead of
   * one per 32-token block.  Forward: S uses K's per-key scales; on the
   * diagonal tile of a causal call, V's per-key exponent is folded into
   * P-hat (its block scale per query row and 32-key group is the largest V
   * exponent among the keys that row sees, less c); the tiles before it hold
   * only keys every row of the tile sees, so they multiply V's token-block
   * codes with the fixed 2^c, as the pages do (a non-causal call has no
   * diagonal tile: every tile uses the token-block codes).  Backward: S and
   * dP use K's and V's per-key scales; dS for dQ carries K's per-key
   * exponent and takes one exponent per (query row, 32-key group); dK's and
   * dV's operands carry Q's and dO's per-token exponents within their
   * 32-query blocks.  No scale then reaches across the causal boundary, so a
   * later token of a document changes no bit of an earlier row's O, LSE or
   * dQ (dQ exactly so within one key tile; across key tiles its fp32
   * reduce-adds may arrive in any order, unless deterministic_dq is set).
   * The saved buffer then holds per-token codes and scales and a
   * token-block copy of V (flamia_saved_bytes_with); pass the same value to
   * both calls.  At d = 128 the backward applies K's and V's per-key
   * exponents to the recomputed S and dP as fp32 column factors (its tensor
   * memory has no room for them as MMA scales); the products are exact, so
   * S and dP round to the same values.  0 = token-block scales (the
   * default). */
  int32_t exact;
  /* How the attention kernels' persistent CTAs share the work list, which is
   * sorted longest-first on the device (FLAMIA Section 3.6.2).  0 = dynamic
   * hand-out (the default): each CTA claims its next item from a counter in
   * the workspace when it has issued its current item's last loads, so the
   * long items start first and every later item goes to the first CTA that
   * needs work.  1 = static: CTA b takes items b, 2G-1-b, 2G+b, ... of the
   * sorted list (G CTAs, alternating direction).  The choice changes which CTA
   * computes an item, never its result: O, LSE, dK and dV are bitwise the
   * same under both. */
  int32_t schedule;
  /* 1 = the mixed NVFP4/FP8 path of FLAMIA Section 3.4.  The forward's
   * scores and their recomputation in the backward multiply NVFP4 Q and K:
   * E2M1 codes with one UE4M3 scale per 16 head-dimension elements of each
   * token (the smallest scale s with 6 s >= the group's largest magnitude;
   * codes are E2M1 round-to-nearest-even of x / s), by a block-scaled 4-bit
   * MMA.  P-hat is quantized in the log domain (Section 3.5.2): each query
   * row and 32-key group takes the round-up exponent of its largest
   * probability as its P-hat scale, and the fixed 2^c_exp is not used.
   * Every other product keeps the E4M3 token-block operands.  The saved
   * buffer then also holds the NVFP4 Q and K (flamia_saved_bytes_with);
   * pass the same value to both calls.  Not combined with exact or hadamard
   * (FLAMIA_ERR_ARG).  0 = MXFP8 scores (the default). */
  int32_t nvfp4;
  /* 1 = a dQ whose bits do not depend on the order in which the backward's
   * key tiles finish (FLAMIA Appendix B.5 on deterministic reductions; the
   * accumulator stays document-local).  Every dQ partial, one per (key tile,
   * query row, channel), is rounded to a signed 64-bit integer count of
   * 2^-32 and added with integer reduce-adds, which are associative, so the
   * same inputs always give bitwise the same dQ, whatever the schedule.  The
   * accumulator is then 8 bytes per element (flamia_workspace_bytes always
   * has room for it).  Limits: a partial or an accumulated value of
   * magnitude 2^31 or more is not represented (partials saturate, sums wrap);
   * partials below 2^-33 in magnitude round to zero.  Costs integer
   * conversions and twice the accumulator traffic in the backward.  The
   * forward does not clear this accumulator, so flamia_bwd zeroes it.  Only
   * flamia_bwd reads this field.  0 = fp32 reduce-adds (the default). */
  int32_t deterministic_dq;
} flamia_opts;

/* Default options: c = 4, tau = 4, causal, no rotation, token-block scales,
 * dynamic hand-out, fp32 dQ reduce-adds. */
flamia_opts flamia_default_opts(void);

/* Bytes of the buffer flamia_fwd fills with the quantized Q, K, V (codes and
 * scale tables) that flamia_bwd reads back, enough for every option.  Layout
 * (each piece 256-byte aligned, in this order): q codes [T,Hq,d], k codes
 * [T,Hkv,d], v codes [T,Hkv,d], q scales [Hq,T], k scales [Hkv,T], v scales
 * [Hkv,T], then the pieces of the NVFP4 or the exact options
 * (flamia_saved_bytes_with gives the size for given options). */
size_t flamia_saved_bytes(int64_t T, int32_t Hq, int32_t Hkv, int32_t d);

/* The same for the given options: with nvfp4 = 1 the buffer continues with
 * the NVFP4 Q and K (each piece 256-byte aligned): q codes [T,Hq,d/2] and k
 * codes [T,Hkv,d/2] (two E2M1 codes per byte, element 2i in the low nibble),
 * q scales [T,Hq,d/16] and k scales [T,Hkv,d/16] (UE4M3 bytes).  With
 * exact = 1 it continues with V quantized with token-block scales: codes
 * [T,Hkv,d] and scales [Hkv,T].  A call with these options needs a buffer of
 * this size.  Returns 0 for an invalid shape or options. */
size_t flamia_saved_bytes_with(int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts);

/* Bytes of scratch memory flamia_fwd / flamia_bwd need ("workspace"): the
 * device-built work lists with their claim counter, the quantized dO and its
 * scales, D, and the dQ accumulator (8 bytes per element of dQ, enough for
 * every option).  It needs no initialization and holds nothing meaningful
 * after a call; calls that run concurrently need separate workspaces. */
size_t flamia_workspace_bytes(int64_t T, int32_t n_docs, int32_t Hq, int32_t Hkv, int32_t d);

/*
 * flamia_quantize - token-block MXFP8 quantization of one packed tensor.
 * (FLAMIA Section 3.1 token-block scaling; Section 3.2 round-up exponent;
 *  Section 3.6.1 document-local blocks on the packed layout.)
 *
 * For every document [s, e), head h and block b, the tokens
 * [s + 32b, min(s + 32b + 32, e)) over all d channels share the exponent E,
 * the smallest integer with max|x| <= 448 * 2^E (clamped to [-127, 127]); the
 * code of x is E4M3(x * 2^-E), round to nearest even, finite saturation.
 *   x_dev       bf16 [T, H, d]             input
 *   codes_dev   uint8 [T, H, d]            output, E4M3 codes
 *   scales_dev  uint8 [H, T]               output, UE8M0 byte per token
 * Tokens outside every document get code 0 and scale byte 0.
 */
int flamia_quantize(const void* x_dev, int64_t T, int32_t H, int32_t d, const int32_t* cu_seqlens_dev,
                    int32_t n_docs, uint8_t* codes_dev, uint8_t* scales_dev, void* stream);

/*
 * flamia_fwd - quantize Q, K, V and run the MXFP8 attention forward.
 * (FLAMIA Sections 3.4-3.6, Appendix B.1.)
 *
 * S = Qhat Khat^T / sqrt(d) per document; online softmax in fp32 over key
 * tiles of 128 document-relative keys (causal: the fully visible tiles from
 * the one below the diagonal down to tile 0, then the diagonal tile;
 * non-causal: the last tile down to tile 0), with the conditional rescale
 * decided per query row; the
 * probabilities are multiplied by 2^c, rounded to E4M3 and multiplied with
 * Vhat by a block-scaled MMA.
 *   q_dev       bf16 [T, Hq, d];  k_dev, v_dev  bf16 [T, Hkv, d]
 *   out_dev     bf16 [T, Hq, d]   output O
 *   lse_dev     float [Hq, T]     output log-sum-exp (natural log); +inf outside documents
 *   saved_dev   flamia_saved_bytes_with(opts) bytes (flamia_saved_bytes() for the default
 *               options), output: quantized Q, K, V for flamia_bwd
 *   work_dev    flamia_workspace_bytes() bytes of scratch.  The forward also
 *               zeroes the fp32 dQ accumulator inside it and stamps it, so a
 *               flamia_bwd given the same workspace skips that zeroing (any
 *               other workspace is zeroed by flamia_bwd itself).
 * The same inputs always give bitwise-identical O and LSE.
 */
int flamia_fwd(const void* q_dev, const void* k_dev, const void* v_dev, const int32_t* cu_seqlens_dev,
               int32_t n_docs, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts,
               void* out_dev, float* lse_dev, void* saved_dev, void* work_dev, void* stream);

/*
 * flamia_fwd_noalloc - flamia_fwd for callers that cannot allocate device
 * memory.  (The paper has no counterpart: this is an integration variant.)
 *
 * Some callers cannot call cudaMalloc when they run attention - code running
 * inside an allocator or memory-pool callback, runtimes that only hand out
 * pre-registered buffers, processes that reserve all device memory up front.
 * This entry point takes the same arguments as flamia_fwd except work_dev and
 * allocates nothing (no cudaMalloc, cudaFree or allocating library call): the
 * forward's only scratch, its device-built work list, lives in a fixed
 * file-scope device array of about 1.6 MB that every GPU which loads the
 * library holds until the process exits.  Results are identical to flamia_fwd.
 *  - Limits: T <= 2^20 tokens and n_docs <= 65536; larger problems are
 *    rejected with FLAMIA_ERR_NOALLOC_LIMIT before any launch.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array: calls that overlap on the
 *    GPU (different streams, or different host threads) race and must be
 *    serialized by the caller.  Each call rewrites the whole work list, so no
 *    state from the previous call is used.
 */
int flamia_fwd_noalloc(const void* q_dev, const void* k_dev, const void* v_dev, const int32_t* cu_seqlens_dev,
                       int32_t n_docs, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts,
                       void* out_dev, float* lse_dev, void* saved_dev, void* stream);

/*
 * flamia_bwd - quantize dO (with D and the dQ accumulator) and run the MXFP8
 * attention backward.  (FLAMIA Sections 2, 3.3, 3.5.3, Appendix B.1.)
 *
 * Reuses the forward's quantized Q, K, V (saved_dev) and recomputes S and P
 * with the forward's S tile, exponential and LSE;  D_i = dOhat_i . O_i with
 * the token-block-quantized dO and the forward output O;  dV = P'^T dOhat
 * with P' = E4M3(2^8 P) 2^-8;  dP = dOhat Vhat^T;  dS = P o (dP - D),
 * quantized in 32x32 blocks;  dQ = dShat Khat / sqrt(d),
 * dK = dShat^T Qhat / sqrt(d).  dK and dV sum over the query heads of a
 * group.
 *   out_dev          bf16 [T, Hq, d]  the forward's output O
 *   lse_dev          float [Hq, T]    the forward's LSE
 *   dout_dev         bf16 [T, Hq, d]  dO
 *   saved_dev        the buffer flamia_fwd filled for these inputs
 *   dq_dev           bf16 [T, Hq, d]  output;  dk_dev, dv_dev  bf16 [T, Hkv, d]  outputs
 *   work_dev         flamia_workspace_bytes() bytes of scratch; its dQ
 *                    accumulator is zeroed here unless the forward of this
 *                    shape stamped it, and the stamp is cleared once the
 *                    accumulator holds sums
 * dK and dV are bitwise reproducible.  By default dQ is accumulated with fp32
 * reduce-adds, so its last bits can vary between runs when a document spans
 * more than one 128-key tile; with opts->deterministic_dq it is bitwise
 * reproducible too.  A score-tile copy (flamia_debug_set_score_dump) is not
 * combined with deterministic_dq (FLAMIA_ERR_UNSUPPORTED_OPT).
 */
int flamia_bwd(const void* out_dev, const float* lse_dev, const void* dout_dev, const int32_t* cu_seqlens_dev,
               int32_t n_docs, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts,
               const void* saved_dev, void* dq_dev, void* dk_dev, void* dv_dev, void* work_dev, void* stream);

/*
 * flamia_get_status - read and clear the device status word of the current
 * device (FLAMIA_STATUS_*).  Synchronizes `stream` (a diagnostic call; not for
 * use inside stream capture).  Returns 0 or FLAMIA_ERR_LAUNCH.
 */
int flamia_get_status(int32_t* status_out, void* stream);

/*
 * flamia_set_launch_events - per-kernel timing hook (no counterpart in the
 * method; measurement plumbing).  `events` points to `n` cudaEvent_t handles
 * created by the caller (n = 0 or events = NULL disables the hook).  While set,
 * every flamia_fwd / flamia_bwd call on this host thread records events[i] on
 * its stream just before its i-th kernel launch and events[L] after the last
 * of its L launches (L = flamia_last_launch_count(), at most n - 1 launches
 * are bracketed).  The events are recorded as external events, so a call made
 * under stream capture puts them into the CUDA graph, where every replay
 * records them again.  Returns 0.
 */
int flamia_set_launch_events(void** events, int32_t n);

/* Number of kernel launches the last successful flamia_fwd / flamia_bwd /
 * flamia_quantize call on this host thread enqueued. */
int32_t flamia_last_launch_count(void);

/*
 * flamia_debug_set_score_dump - diagnostic (no counterpart in the method).
 * While set, flamia_fwd and flamia_bwd calls on this host thread run variants
 * of the attention kernels that also copy out one score tile, so that a test
 * can check that the backward recomputes the forward's S tile bit for bit
 * (FLAMIA Section 3.3: the backward reuses the forward's quantized
 * representation, tiling and exponential).  The tile is (query head h,
 * document doc, query tile qt, key tile kt), tiles counting 128
 * document-relative tokens; the call must visit it (causal: kt <= qt).
 *   s_fwd_dev, s_bwd_dev  float [128][128] outputs: the raw fp32 accumulator
 *                         of Qhat Khat^T on the E4M3 codes (row = query,
 *                         column = key), before any mask
 *   f_fwd_dev, f_bwd_dev  float [128][4] outputs: per query row and 32-key
 *                         group, the factor 2^(E_Q + E_K) log2(e)/sqrt(d)
 *                         the kernel applies to those accumulators
 * Rows or keys past the document end hold what the tile computes there.  A
 * null s_fwd_dev (s_bwd_dev) leaves the forward (backward) on its normal
 * kernels; all four null disables the hook.  Token-block scales only: while a
 * copy is requested, a call with the exact options returns
 * FLAMIA_ERR_UNSUPPORTED_OPT.  Returns 0.
 */
int flamia_debug_set_score_dump(float* s_fwd_dev, float* f_fwd_dev, float* s_bwd_dev, float* f_bwd_dev, int32_t h,
                                int32_t doc, int32_t qt, int32_t kt);

/*
 * flamia_debug_set_item_limit - diagnostic (no counterpart in the method): a
 * way to make the on-chip wait timeout happen on purpose, so that a test can
 * check how a call that gives up ends.  While n > 0, every flamia_fwd call on
 * this host thread runs with each persistent CTA handing out at most n work
 * items (FLAMIA Section 3.6.2's work list): after its n-th item the CTA's
 * producer issues nothing more, not even the end-of-work marker, and lets its
 * in-flight copies land.  The CTA's other warps finish their items, wait for
 * the next one until the wait budget (about 2 s) runs out, report
 * FLAMIA_STATUS_TIMEOUT and wind down (their tensor-core work completes
 * before tensor memory is freed).  The outputs of such a call are
 * incomplete; later calls are unaffected.  n = 0 (the default) turns the
 * limit off.  Returns 0, or FLAMIA_ERR_ARG for n < 0.
 */
int flamia_debug_set_item_limit(int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* FLAMIA_H_ */
