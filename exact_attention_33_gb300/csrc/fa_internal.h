// fa_internal.h - parameter blocks and constants shared by the host glue
// (fa_api.cu) and the kernels.  Plain structs passed to kernels by value.
#pragma once

#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

// Bound for every on-chip spin-wait (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Control block at the start of a decode or split-KV workspace (its first
// FA_WORKSPACE_HEADER_BYTES bytes).  Zero before the first call that uses
// the workspace; every call leaves acc at zero again.
struct CallStatus {
  unsigned int acc;   // FA_DEV_* bits raised by the call in flight
  unsigned int last;  // FA_DEV_* bits of the last call that finished
};
static_assert(sizeof(CallStatus) <= FA_WORKSPACE_HEADER_BYTES, "workspace header too small");

// ------------------------------------------------------------------ prefill

// Tile shape of the prefill kernel: each CTA owns two 128-row query tiles
// (one per softmax warpgroup) of one (sequence, head) and streams 128-key
// K/V tiles through shared memory.
constexpr int kPrefillBM = 128;
constexpr int kPrefillBN = 128;
constexpr int kPrefillQTiles = 2;
constexpr int kPrefillRowsPerCta = kPrefillBM * kPrefillQTiles;
constexpr int kPrefillThreads = 352;  // 8 softmax warps, 1 MMA warp, 2 TMA warps

// The same kernel with one query tile per CTA (packed batches of short
// sequences): 256 threads, warps 0-3 softmax, 4 MMA, 5 and 6 TMA, 7 idle, and two
// CTAs per SM, so that one CTA's launch, set-up and epilogue overlap the
// other's key loop.  Each CTA is built for 128 registers per thread and moves
// them with setmaxnreg: the softmax warpgroup up to 168, the other down to 88
// (4 * 32 * 168 + 4 * 32 * 88 = 256 * 128; per SMSP, two CTAs use 2 * 32 *
// 168 + 2 * 32 * 88 = 16384, the SMSP's register file).
constexpr int kPrefill1LaunchRegs = 128;
constexpr int kPrefill1SoftmaxRegs = 168;
constexpr int kPrefill1CtlRegs = 88;
static_assert(128 * kPrefill1SoftmaxRegs + 128 * kPrefill1CtlRegs <= 256 * kPrefill1LaunchRegs,
              "one-tile prefill register split exceeds the launch allocation");

// Shape of a prefill CTA with QT query tiles.
template <int QT>
struct PrefillShape {
  static_assert(QT == 1 || QT == 2, "one or two query tiles per CTA");
  static constexpr int kRows = kPrefillBM * QT;
  static constexpr int kThreads = QT == 2 ? kPrefillThreads : 256;
  static constexpr int kSoftmaxWarps = 4 * QT;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static constexpr int kTmaWarp = kSoftmaxWarps + 1;   // Q and K/V copies (K only when paged)
  static constexpr int kTmaVWarp = kSoftmaxWarps + 2;  // V copies of a paged KV cache
  static constexpr int kMinBlocks = QT == 2 ? 1 : 2;
};

// Work layouts of the prefill kernel.
constexpr int kKindDense = 0;   // [B, N, H, d] batch
constexpr int kKindVarlen = 1;  // packed sequences, cu_seqlens
constexpr int kKindPaged = 2;   // packed query chunks over a paged KV cache
constexpr int kKindDenseSplit = 3;  // dense batch, key tiles split over CTAs
constexpr int kKindVarlenHeads = 4;  // packed sequences; a CTA's two query tiles are two heads
                                     // of one KV group over the same 128 rows
constexpr int kKindDenseHeads = 5;   // dense batch, the same head pairs
constexpr int kKindPagedHeads = 6;   // paged KV cache, the same head pairs

// Packed batches of at most this many sequences use the padding-free order
// of work items (each CTA finds its item with one pass over cu_seqlens).
constexpr int kVarlenCompactMaxSeqs = 128;

struct PrefillParams {
  // FA_DEV_* bits go to `status`: the per-device sticky word, or for a call
  // with a workspace its accumulator, which the call's last kernel publishes
  // (into the control block and the per-device word dev_status).
  unsigned int *status;
  CallStatus *call;           // control block of the call's workspace, or null
  unsigned int *dev_status;   // per-device sticky word
  void *out;              // bf16 [rows, H, d] (dense rows = B*N, varlen rows = T)
  float *lse;             // fp32, may be null
  const int32_t *cu_seqlens;  // varlen only
  int B;                  // dense: batch; varlen: number of sequences
  int H, Hkv, group;      // group = H / Hkv
  int head_group;         // heads per CTA-ordering group (divides H)
  int N;                  // dense: sequence length; varlen: total tokens
  int max_pairs;          // number of 256-row query-tile pairs of the longest sequence
  int compact;            // varlen: work items enumerate only real (sequence, pair) items
  int total_tokens;       // varlen: T
  float scale_log2;       // scale * log2(e) (times the q and k descales for fp8)
  float v_descale;        // multiplies the output (1 for bf16)
  int causal;
  // dense and packed kinds: each CTA prefetches into L2 the Q tiles of work
  // item (its own + prefetch_ahead), the one that starts about a wave later
  // (0: none)
  int prefetch_ahead;
  // split kind only: partial states
  int num_splits;
  float *o_part;   // fp32 [splits, B, N, H, d]
  float *ml_part;  // fp32x4 [splits, B, N, H]: m (log2 units), l, l_exact, 0
  // paged kind only
  const int32_t *block_table;  // [num_seqs, max_blocks_per_seq]
  const int32_t *ctx_lens;     // keys per sequence
  int max_blocks_per_seq;
  int max_ctx_len;
  int num_blocks;
};

// ------------------------------------------------------------------- decode

constexpr int kDecodeBlock = 16;     // tokens per KV block (paged pool granularity)
constexpr int kDecodeStages = 4;     // KV blocks in flight per CTA
constexpr int kCombineWarps = 4;
constexpr int kDecodeMaxSplitTokens = 512;  // one block-table entry per lane of the split warp

struct DecodeParams {
  unsigned int *status;       // the workspace's accumulator of FA_DEV_* bits
  CallStatus *call;           // control block of the call's workspace
  unsigned int *dev_status;   // per-device sticky word
  const void *q;            // bf16 [batch, H, d]
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *o_part;            // fp32 [batch, H, max_splits, d]
  float *ml_part;           // fp32 [batch, H, max_splits, 2]  (m in log2 units, l)
  void *out;                // bf16 [batch, H, d]
  float *lse;               // fp32 [batch, H] or null
  int batch, H, Hkv, group;
  int max_blocks_per_seq;
  int max_ctx_len;
  int num_blocks;
  int split_tokens;         // multiple of kDecodeBlock
  int max_splits;
  float scale_log2;
};

}  // namespace fa
