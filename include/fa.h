/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * Exact scaled-dot-product attention computed as a tiled, IO-aware
 * streaming recurrence: key/value tiles are staged on chip, the score tile
 * S = scale * Q K^T is formed per tile and never written to device memory,
 * and the softmax is folded in online with a running row maximum m, a
 * running sum l and the rescale factor alpha = exp(m_old - m_new); the
 * output accumulator o is finished as o / l.
 *   Sources: "S12 FlashAttention" (llminference.xinbetween.com/en/s12/),
 *   sections "Core idea", "How it works" (the recurrence diagram),
 *   "What this unlocks beyond speed" and "Implementation"; the FlashAttention
 *   explainer (tachyon.techntrek.in/learn/flash-attention), "Show the maths";
 *   and "FlashAttention: The Algorithm That Beat the Memory Wall"
 *   (repo-explainer.com/hillfate/flash-attention), sections "A Tile, a
 *   Register File, and a Trick Called Online Softmax" and "Varlen Is the
 *   Quiet Superpower".
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor arguments are DEVICE pointers owned by the caller; the
 *    library never allocates, frees or synchronises on the compute path.
 *    Every call is asynchronous on `stream` (NULL = legacy default stream).
 *  - bf16 = IEEE bfloat16; fp32 accumulation; outputs are rounded to
 *    bf16 (round to nearest even), the log-sum-exp is fp32.
 *  - Element layouts are dense row-major with the innermost dimension last;
 *    q/k/v/out and pools must be 16-byte aligned (TMA requirement).
 *  - GQA: query head h reads key/value head h / (H / Hkv).
 *  - `scale` multiplies q.k before the softmax; it must be finite and > 0
 *    (the usual value is 1/sqrt(d)).
 *  - lse (optional, may be NULL) receives the natural-log log-sum-exp of the
 *    scaled scores of each query row: LSE = m + ln(l).
 *  - Return value: FA_OK, or a negative fa_status.  Argument errors are
 *    detected on the host before any launch and launch nothing.  Launch
 *    failures return FA_ERR_CUDA.  Data errors that only the device can see
 *    (an out-of-range block id, a bad context length, a pipeline wait that
 *    ran out of time) set bits of a per-device sticky status word that
 *    fa_device_status() reads; the affected work is skipped, never trapped.
 *    Calls that take a workspace (fa_decode_paged, fa_fwd_splitkv) record
 *    their bits in the workspace, where fa_last_device_status() reads them
 *    without touching other streams' work, and add them to the per-device
 *    word when they finish.
 *  - Workspaces: the first FA_WORKSPACE_HEADER_BYTES bytes of a decode or
 *    split-KV workspace are the call's control block (the bits its kernels
 *    raise, and the status of the last call that finished).  Zero-fill a
 *    new workspace once before its first call (cudaMemsetAsync,
 *    torch.zeros); every call leaves the block ready for the next.  Calls that share a workspace must
 *    be ordered (one stream, or events); calls on different workspaces are
 *    independent.
 *  - The library caches per-device addresses of its own device variables;
 *    do not keep using it in a process after cudaDeviceReset().
 *  - Supported head sizes: d in {64, 128}.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misalignment, H % Hkv != 0 ... */
  FA_ERR_UNSUPPORTED = -2, /* valid request outside what is built (e.g. d = 96)      */
  FA_ERR_CUDA = -3,        /* a CUDA runtime/driver call or a launch failed          */
  FA_ERR_WORKSPACE = -4    /* decode workspace missing, misaligned or too small      */
} fa_status;

/* Bytes at the start of a decode or split-KV workspace that hold the
   call's control block (included in the workspace sizes below). */
#define FA_WORKSPACE_HEADER_BYTES 256u

/* Bits of the per-device sticky status word. */
#define FA_DEV_TIMEOUT 1u     /* a bounded on-chip pipeline wait gave up             */
#define FA_DEV_BAD_BLOCK 2u   /* block_table entry outside [0, num_blocks)           */
#define FA_DEV_BAD_CTX 4u     /* ctx_len < 0 or > max_blocks_per_seq * block_size    */
#define FA_DEV_BAD_SEQLEN 8u  /* cu_seqlens not non-decreasing / beyond total_tokens */
#define FA_DEV_BAD_INDEX 16u /* checked build only: a kernel index outside its buffer  */
#define FA_DEV_SMEM_ALIGN 32u /* a kernel found its shared memory not 1 KiB aligned    */

/*
 * Dense prefill forward (causal or not).
 *   q, out : [B, N, H, d]   bf16
 *   k, v   : [B, N, Hkv, d] bf16
 *   lse    : [B, H, N]      fp32, may be NULL
 *   causal : 0 or 1; masking is bottom-right aligned (key j visible to query
 *            i iff j <= i + (Nk - Nq)), which is j <= i here since Nq = Nk.
 * The recurrence of "S12 FlashAttention" ("Core idea"; exercise 2 for the
 * causal variant) over tiles of 128 keys, for tiles of 128 query rows.
 * B == 0 or N == 0 is a no-op.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
           int B, int H, int Hkv, int N, int d, float scale, int causal,
           fa_stream_t stream);

/*
 * Packed variable-length prefill ("Varlen Is the Quiet Superpower"): the
 * sequences are concatenated along the token axis with no padding.
 *   q, out     : [total_tokens, H, d]   bf16
 *   k, v       : [total_tokens, Hkv, d] bf16
 *   lse        : [H, total_tokens]      fp32, may be NULL
 *   cu_seqlens : int32 DEVICE array [num_seqs + 1], non-decreasing,
 *                cu_seqlens[0] == 0, cu_seqlens[num_seqs] == total_tokens.
 *   max_seqlen : an upper bound of every sequence length (sizes the launch).
 * Sequence s attends only to its own tokens [cu[s], cu[s+1]); the causal
 * rule applies per sequence.  Work items are (sequence, q-tile, head) with
 * no padding tiles.  A cu_seqlens array that breaks the rules above sets
 * FA_DEV_BAD_SEQLEN and the offending sequence is skipped.
 */
int fa_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                  const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                  int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                  fa_stream_t stream);

/*
 * Dense prefill with FP8 (e4m3) inputs on the kind::f8f6f4 tensor-core path
 * ("S12 FlashAttention", Production notes: the Hopper generation of the
 * method adds FP8 support).  q, k, v hold e4m3 codes (one byte each) in the
 * layouts of fa_fwd; the real values are code * q_descale, code * k_descale,
 * code * v_descale (per-tensor, finite, > 0).  The softmax weights P are
 * rounded to e4m3 for the P V product, so the output error is bounded by
 * about 2^-4 times the attention-weighted mean of |v| (see the tests).
 *   out : [B, N, H, d] bf16;  lse : [B, H, N] fp32, may be NULL
 * Supported: d == 64 or 128 (other d: FA_ERR_UNSUPPORTED).
 */
int fa_fwd_fp8(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
               int Hkv, int N, int d, float scale, float q_descale, float k_descale,
               float v_descale, int causal, fa_stream_t stream);

/*
 * Packed variable-length prefill with FP8 (e4m3) inputs: the layouts and
 * sequence rules of fa_fwd_varlen ("Varlen Is the Quiet Superpower"), the
 * codes and per-tensor descales of fa_fwd_fp8.
 *   q          : [total_tokens, H, d]   e4m3 codes (one byte each)
 *   k, v       : [total_tokens, Hkv, d] e4m3 codes
 *   out        : [total_tokens, H, d]   bf16;  lse : [H, total_tokens] fp32, may be NULL
 *   cu_seqlens : int32 DEVICE array [num_seqs + 1] (rules as fa_fwd_varlen)
 * Supported: d == 64 or 128.  Errors as fa_fwd_varlen and fa_fwd_fp8.
 */
int fa_fwd_varlen_fp8(const void *q, const void *k, const void *v, void *out, float *lse,
                      const int32_t *cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                      int H, int Hkv, int d, float scale, float q_descale, float k_descale,
                      float v_descale, int causal, fa_stream_t stream);

/*
 * Gradient of dense attention (backward pass): given the forward inputs, its
 * output O and log-sum-exp, and the upstream gradient dO, writes
 *   dV = P^T dO,  dQ = scale dS K,  dK = scale dS^T Q,
 *   dS = P * (dO V^T - rowsum(dO * O)),  P = exp(scale Q K^T - lse)
 * (masked entries 0), summed over the query heads of each KV head.  The pages
 * describe only the forward streaming softmax ("S12 FlashAttention"); this
 * is the chain rule through that definition, with P recomputed tile by tile
 * from Q, K and the forward log-sum-exp instead of being stored.  No
 * gradient flows through the log-sum-exp output.
 *   q, out, dout, dq : [B, N, H, d] bf16     k, v, dk, dv : [B, N, Hkv, d] bf16
 *   lse              : [B, H, N] fp32, as written by fa_fwd (same q, k, v,
 *                      scale and causal flag)
 *   workspace        : caller-owned device memory of at least
 *                      fa_bwd_workspace_size(B, H, N) bytes, 256-byte aligned;
 *                      overwritten (fp32 rowsums and rescaled lse, then the
 *                      work counters of the two persistent gradient kernels,
 *                      which the call zeroes itself); one call at a time per
 *                      workspace
 * Supported: d in {64, 128}.  All buffers device memory; asynchronous on
 * `stream`.  Errors as for fa_fwd; FA_ERR_WORKSPACE for a missing, small or
 * misaligned workspace.
 */
size_t fa_bwd_workspace_size(int B, int H, int N);
int fa_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int N, int d,
           float scale, int causal, void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Gradient of a packed batch of variable-length sequences: the fa_bwd
 * products applied to each sequence of an fa_fwd_varlen call on its own rows
 * (its keys are the only ones its queries see; causal masking by position
 * inside the sequence).  The same definition as fa_bwd (chain rule through
 * "S12 FlashAttention"'s softmax), with the packing of fa_fwd_varlen.
 *   q, out, dout, dq : [total_tokens, H, d] bf16
 *   k, v, dk, dv     : [total_tokens, Hkv, d] bf16
 *   lse              : [H, total_tokens] fp32, as written by fa_fwd_varlen
 *   cu_seqlens       : int32 DEVICE array [num_seqs + 1]; sequence s is rows
 *                      [cu_seqlens[s], cu_seqlens[s + 1]).  A sequence whose
 *                      bounds are decreasing, outside [0, total_tokens] or
 *                      longer than max_seqlen raises FA_DEV_BAD_SEQLEN and its
 *                      rows of dq, dk and dv are not written; rows that belong
 *                      to no sequence are not written either.
 *   max_seqlen       : upper bound on every sequence's length
 *   workspace        : >= fa_bwd_workspace_size(num_seqs, H, max_seqlen)
 *                      bytes, 256-byte aligned, owned by the caller;
 *                      overwritten
 * Supported: d in {64, 128}.  All buffers device memory; asynchronous on
 * `stream`.  Errors as fa_bwd.
 */
int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *out, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, const int32_t *cu_seqlens,
                  int num_seqs, int total_tokens, int max_seqlen, int H, int Hkv, int d,
                  float scale, int causal, void *workspace, size_t workspace_bytes,
                  fa_stream_t stream);

/*
 * Dense prefill with the key tiles of every query tile split over several
 * CTAs, for batches whose B * H * ceil(N / 256) work items cannot fill the
 * GPU (long single sequences).  "S12 FlashAttention", "What this unlocks
 * beyond speed": the same recurrence applied across processors - each split
 * produces a partial (m, l, o) state and a second kernel merges them with the
 * rescaling of the explainer page's "Show the maths".
 * Arguments and results as fa_fwd, plus:
 *   num_splits : 1..16, or 0 to let the library choose (about 1.7 CTAs per
 *                SM: 2 splits for 128 work items on 152 SMs, 1 from about
 *                152 work items up); values above the number of 128-key
 *                tiles are clamped.
 *   workspace  : >= fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
 *                bytes, 256-byte aligned, owned by the caller, zero-filled
 *                before its first call (the control block).
 * Two kernels run in stream order: the split prefill and the combine.  With
 * one split the call runs the fa_fwd kernel (no partial states) and a
 * one-warp kernel that publishes the call's status in the workspace.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits);
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                   int H, int Hkv, int N, int d, float scale, int causal, int num_splits,
                   void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Prefill of query chunks against a paged KV cache (chunked prefill / cached
 * prefix): "S12 FlashAttention", "Implementation" - the paged variant is the
 * same tiled recurrence with the block table in front of the key access.
 * Each sequence b brings cu_seqlens_q[b+1] - cu_seqlens_q[b] query tokens
 * (packed as in fa_fwd_varlen) and reads its ctx_lens[b] keys, the cached
 * prefix plus the chunk itself, which the caller has already written to the
 * pool.
 *   q, out       : [total_q, H, d] bf16
 *   k_pool,
 *   v_pool       : [num_blocks, block_size, Hkv, d] bf16, block_size == 16
 *   block_table  : int32 [batch, max_blocks_per_seq]
 *   ctx_lens     : int32 [batch], 0 <= ctx_lens[b] <= max_ctx_len
 *   cu_seqlens_q : int32 DEVICE array [batch + 1] (rules as cu_seqlens)
 *   lse          : [H, total_q] fp32, may be NULL
 *   causal       : bottom-right aligned: query i of a chunk of Nq queries
 *                  sees key j iff j <= i + (ctx_len - Nq).  A query that sees
 *                  no key gets out = 0 and lse = -inf.
 * Slots of the last block past ctx_len are never copied on chip.  Device-side
 * checks: FA_DEV_BAD_CTX, FA_DEV_BAD_BLOCK, FA_DEV_BAD_SEQLEN.
 */
int fa_fwd_paged(const void *q, const void *k_pool, const void *v_pool,
                 const int32_t *block_table, int max_blocks_per_seq, const int32_t *ctx_lens,
                 const int32_t *cu_seqlens_q, int batch, int total_q, int max_seqlen_q,
                 int max_ctx_len, int H, int Hkv, int d, int block_size, int num_blocks,
                 float scale, int causal, void *out, float *lse, fa_stream_t stream);

/*
 * Bytes of caller-owned workspace that fa_decode_paged needs: the control
 * block plus the split partial states (m, l, o) of every (sequence, query
 * head, key split).  Returns 0 for invalid arguments.  The split size
 * depends only on these arguments and on the current device's SM count; Hkv
 * is among them because the number of splits is chosen so that the
 * (sequence, KV head, split) work items fill the GPU.
 */
size_t fa_decode_workspace_size(int batch, int H, int Hkv, int d, int max_ctx_len,
                                int block_size);

/*
 * Paged GQA flash-decoding: one query token per sequence against a paged
 * KV cache ("S12 FlashAttention": "Implementation" - the block table in front
 * of the key access; "What this unlocks beyond speed" - split the keys across
 * thread blocks and combine the partial (m, l, o) states; "How this composes
 * with what you already built" - paging, GQA head sharing and the recurrence
 * in one loop).
 *   q, out      : [batch, H, d] bf16
 *   k_pool,
 *   v_pool      : [num_blocks, block_size, Hkv, d] bf16
 *   block_table : int32 [batch, max_blocks_per_seq]; logical block j of
 *                 sequence b is physical block block_table[b][j]
 *   ctx_lens    : int32 [batch], 0 <= ctx_lens[b] <= max_ctx_len
 *   lse         : [batch, H] fp32, may be NULL
 *   workspace   : >= fa_decode_workspace_size(...) bytes, 256-byte aligned,
 *                 owned by the caller; zero-filled before its first call
 *                 (the control block, see the conventions above); past the
 *                 control block its contents on entry are ignored.
 * A sequence with ctx_len 0 gets out = 0 and lse = -inf.  Slots of the last
 * block past ctx_len are never read into the result.  Supported: block_size
 * == 16, H / Hkv <= 16.  Two kernels run in stream order: the split kernel
 * and the (m, l, o) combine.
 */
int fa_decode_paged(const void *q, const void *k_pool, const void *v_pool,
                    const int32_t *block_table, int max_blocks_per_seq,
                    const int32_t *ctx_lens, int max_ctx_len, int batch, int H,
                    int Hkv, int d, int block_size, int num_blocks, float scale,
                    void *out, float *lse, void *workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/*
 * Paged decode that allocates nothing and takes no workspace.
 * The pages have no counterpart of this call; it exists for callers that
 * cannot call cudaMalloc: for example a C plugin run by a host framework that
 * owns every device allocation and hands the plugin only its input and output
 * buffers, or a latency-critical decode loop that must not pay the implicit
 * device synchronisation of cudaMalloc/cudaFree.
 * Same arguments, layouts and results as fa_decode_paged, minus the
 * workspace.  The split partial states live in a library-owned static device
 * array of FA_DECODE_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads
 * the library holds until the process exits.
 *  - A request whose partial states would need more than that (compare
 *    fa_decode_workspace_size() with FA_DECODE_NOALLOC_SCRATCH_BYTES) returns
 *    FA_ERR_WORKSPACE and launches nothing.
 *  - The first call on a device looks up the array's device address on that
 *    device (with it current); make that first call before any stream
 *    capture.
 *  - Every call on a device shares the one array and it keeps the last call's
 *    contents.  Only its first FA_WORKSPACE_HEADER_BYTES bytes (the control
 *    block of fa_decode_paged) must start at zero: the array is zero when the
 *    library is loaded, and every call leaves that block at zero again.  The
 *    partial states need no clearing, because each call writes every one of
 *    them before its combine reads it.  Calls whose kernels overlap on the
 *    GPU (other streams, other host threads) race on the array and must be
 *    ordered by the caller.  Device-side errors of these calls are read with
 *    fa_device_status().
 */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
int fa_decode_paged_noalloc(const void *q, const void *k_pool, const void *v_pool,
                            const int32_t *block_table, int max_blocks_per_seq,
                            const int32_t *ctx_lens, int max_ctx_len, int batch, int H,
                            int Hkv, int d, int block_size, int num_blocks, float scale,
                            void *out, float *lse, fa_stream_t stream);

/* Human-readable text of an fa_status value (static storage). */
const char *fa_status_string(int status);

/*
 * Device-side status of the last call that finished on `workspace` (a
 * fa_decode_paged or fa_fwd_splitkv workspace): its FA_DEV_* bits (>= 0; 0 =
 * no device-side error), or a negative fa_status if the read failed.  The
 * pages state the problem with the caller owning every buffer; this is the
 * status word of the call's own workspace, so concurrent callers on other
 * workspaces and streams neither see nor clear each other's errors.
 * Read it after the call has completed (the caller synchronises its own
 * stream or event first); the read is a 4-byte device-to-host copy on the
 * calling thread's per-thread default stream and does not wait for other
 * streams.  Before any call has finished on a zero-filled workspace it
 * returns 0.  A call that launches nothing (an empty problem) leaves the
 * word unchanged.  The index checks of the checked build's combine kernels
 * report to the per-device word only.
 */
int fa_last_device_status(const void *workspace);

/*
 * Read the sticky device status word of the current device into *status
 * (FA_DEV_* bits; 0 = no device-side error since the last clear) and clear
 * it when `clear` != 0.  It gathers the bits of every call on the device,
 * with or without a workspace.  This call synchronises the device.
 */
int fa_device_status(unsigned int *status, int clear);

/*
 * Self-test of the failure path: launches one warp that waits, through the
 * library's bounded pipeline wait, on a barrier that nothing completes.  The
 * wait gives up after about one second, sets FA_DEV_TIMEOUT in the status
 * word and writes 0 to *wait_result (a DEVICE int; 1 would mean the wait
 * succeeded).  The context stays usable.  Asynchronous on `stream`.
 */
int fa_selftest_wait_timeout(int *wait_result, fa_stream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
