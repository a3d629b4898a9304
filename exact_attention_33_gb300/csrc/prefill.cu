// prefill.cu - exact-attention prefill forward for sm_103a.
//
// The streaming recurrence of "S12 FlashAttention" ("Core idea", and the
// recurrence diagram under "How it works"): for each key tile,
//   m_new = max(m, rowmax(s)),  alpha = exp(m - m_new),  p = exp(s - m_new),
//   l = alpha * l + rowsum(p),  o = alpha * o + p V,
// finished as o / l.  The tile arithmetic follows the tiled pseudocode of
// "FlashAttention: The Algorithm That Beat the Memory Wall" ("A Tile, a
// Register File, and a Trick Called Online Softmax"), with the unnormalised
// accumulator of the first page (one division at the end).
//
// GB300 mapping (one CTA = two 128-row query tiles of one (sequence, head)):
//   warp 9      TMA producer: Q tiles once, then K/V tiles of 128 keys into
//               rings of shared-memory stages (128-byte swizzle).  With a
//               paged KV cache, whose copies go block by block through the
//               block table, warp 9 copies the K tiles and warp 10 the V
//               tiles.
//   warp 8      MMA issuer (one thread): S_i = Q_i K^T and O_i += P_i V on the
//               5th-generation tensor cores, fp32 accumulators in TMEM.
//   warps 0-7   two softmax warpgroups, one per query tile; thread t owns
//               query row t of its tile (TMEM lane t).  Each reads its S row
//               from TMEM, applies the mask, updates (m, l), writes P (bf16)
//               back into TMEM over S for the P V product, rescales O by alpha
//               in TMEM, and finally writes O / l and the log-sum-exp.
// The score tile lives only in TMEM and registers; it never reaches HBM.
// Exponentials are taken in base 2 with log2(e) folded into the scale.
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256, 256+d), O_1 after it.
// P_i (bf16, two per column) occupies the first 64 columns of S_i.
//
// With one query tile per CTA (template QT = 1, used for packed batches of
// short sequences) the same roles run as warps 0-3 (softmax), 4 (MMA) and 5
// (TMA) of 256 threads, with S_0 [0,128) and O_0 [128, 128+d) in 256 TMEM
// columns and one K and one V stage at d = 128, so two CTAs share an SM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "checks.cuh"

namespace fa {

// The reference maximum of the exponentials moves only when the row maximum
// grows by more than this many powers of two.
constexpr float kRescaleLog2 = 8.f;



template <int D, bool FP8 = false, int QT = 2>
struct PrefillLayout {
  static constexpr int kElemBytes = FP8 ? 1 : 2;
  // Rows are copied and read in swizzled rows of 128 bytes, or of 64 bytes
  // when a whole row is that short (e4m3 at d = 64: the 64-byte swizzle).
  static constexpr int kSwz = (D * kElemBytes < 128) ? D * kElemBytes : 128;
  static constexpr int kChunkElems = kSwz / kElemBytes;  // elements per swizzled row
  static constexpr int kChunkBytes = 128 * kSwz;         // 128 rows x one swizzled row
  static constexpr int kChunks = D * kElemBytes / kSwz;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kSbo = 8 * kSwz;                  // bytes per 8-row core matrix group
  static_assert(kSwz == 128 || kSwz == 64, "128- or 64-byte rows");
  // K and V have rings of their own: a K stage is released as soon as both
  // S MMAs have read it, a V stage after both P V MMAs.
#ifndef FA_PREFILL_STAGES_K128
#define FA_PREFILL_STAGES_K128 3
#define FA_PREFILL_STAGES_V128 2
#endif
  // With one query tile per CTA two CTAs share an SM's shared memory, so
  // 32 KiB tiles get one stage each.
  static constexpr int kStagesK =
      (QT == 1) ? ((kTileBytes == 32768) ? 1 : 2) : ((kTileBytes == 32768) ? FA_PREFILL_STAGES_K128 : 5);
  static constexpr int kStagesV =
      (QT == 1) ? ((kTileBytes == 32768) ? 1 : 2) : ((kTileBytes == 32768) ? FA_PREFILL_STAGES_V128 : 5);
  // Row sums on the tensor cores (d = 64): the P V product also multiplies
  // P by a block of ones (16 columns of 1.0 beside each V tile, through the
  // descriptor's leading-byte offset), so column D of O accumulates the sum
  // of the bf16 weights of each row, rescaled with O.  O then takes D + 16
  // TMEM columns (2 x (128 + 80) <= 512); at d = 128 there is no room.
  static constexpr bool kOnes = (D == 64) && !FP8;
  static constexpr int kOCols = kOnes ? D + 16 : D;  // TMEM columns of O
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + QT * kTileBytes;
  static constexpr int kV = kK + kStagesK * kTileBytes;
  static constexpr int kOnesOff = kV + kStagesV * kTileBytes;  // 128 x 64 bf16 ones (one chunk)
  static constexpr int kBar = kOnesOff + (kOnes ? kChunkBytes : 0);
  // q_full, k_full[SK], k_empty[SK], v_full[SV], s_full[2], p_full[2],
  // o_done[2], drain, v_empty[SV].  A V stage is released as soon as the
  // P V products of its key tile are done.
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 7;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;     // base is aligned up to 1024 in-kernel
  static constexpr uint32_t kTmemCols = QT * 256;
  // TMEM columns: S_i at 128 i (P_i over its first columns), O_i at
  // kTmemO + kOCols i.
  static constexpr int kTmemO = QT * 128;
};

// Work item `lin` of the padding-free order of a packed batch: sequences in
// order; inside a sequence, groups of p.head_group heads; inside a group the
// pair index varies slowest (heaviest first when causal) and the head
// fastest.  A sequence of len rows owns H * ceil(len / 256) items, so the
// grid needs no item per (sequence, pair) that has no rows.  Every warp
// finds its item with one pass over cu_seqlens, 32 sequences at a time
// (all lanes active).  Returns false past the last item.  Items count ROWS
// query rows by HSTEP heads (h is the first of them).
template <int ROWS, int HSTEP>
__device__ __forceinline__ bool varlen_compact_item(const PrefillParams &p, int lin, bool causal,
                                                    int &unit, int &pair, int &h) {
  const int lane = threadIdx.x & 31;
  if (lin == 0 && threadIdx.x < 32) {
    // A sequence with invalid bounds owns no item here; CTA 0 reports it.
    for (int s = lane; s < p.B; s += 32) {
      const int a = checked_load(p.cu_seqlens, s, p.B + 1, p.status);
      const int e = checked_load(p.cu_seqlens, s + 1, p.B + 1, p.status);
      if (a < 0 || e < a || e > p.total_tokens) raise_status(p.status, FA_DEV_BAD_SEQLEN);
    }
  }
  int base = 0;
  for (int s0 = 0; s0 < p.B; s0 += 32) {
    const int s = s0 + lane;
    int np = 0;
    if (s < p.B) {
      const int a = checked_load(p.cu_seqlens, s, p.B + 1, p.status);
      const int e = checked_load(p.cu_seqlens, s + 1, p.B + 1, p.status);
      const int n = min(max(e - a, 0), p.total_tokens);
      np = (n + ROWS - 1) / ROWS;
    }
    const int mine = np * (p.H / HSTEP);  // items of sequence s
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lin < base + total) {
      const int l = __ffs(__ballot_sync(0xffffffffu, lin < base + incl)) - 1;
      unit = s0 + l;
      const int lu = lin - base - __shfl_sync(0xffffffffu, incl - mine, l);
      const int nps = __shfl_sync(0xffffffffu, np, l);
      const int hgs = p.head_group / HSTEP;  // head slots per ordering group
      const int rem = lu % (hgs * nps);
      h = ((lu / (hgs * nps)) * hgs + rem % hgs) * HSTEP;
      pair = causal ? (nps - 1 - rem / hgs) : rem / hgs;
      return true;
    }
    base += total;
  }
  return false;
}

// KIND: dense batch, packed varlen batch, or packed queries over a paged KV
// cache (chunked prefill).
template <int D, bool CAUSAL, int KIND, bool FP8 = false, int QT = 2>
__global__ void __launch_bounds__(PrefillShape<QT>::kThreads, PrefillShape<QT>::kMinBlocks)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_v1,
                   const __grid_constant__ CUtensorMap tm_o, const PrefillParams p) {
  using L = PrefillLayout<D, FP8, QT>;
  using Sh = PrefillShape<QT>;
  static_assert(!(FP8 && KIND == kKindDenseSplit), "the split-KV layout is bf16 only");
  constexpr int SK = L::kStagesK;
  constexpr int SV = L::kStagesV;
  // the combine of a split launch may be scheduled once every split CTA has started
  if constexpr (KIND == kKindDenseSplit) pdl_launch_dependents();

  // ---------------------------------------------------------- work item
  // One CTA per (sequence, 256-row query pair, head).  CTAs are ordered in
  // groups of p.head_group heads of one sequence: inside a group the pair
  // index varies slowest and the head fastest, so the CTAs running at the
  // same time share the K/V of a few heads in L2.  For causal attention the
  // pairs with the most key tiles come first in every group.
  // Split-KV layout: the split index varies fastest; each split owns a
  // contiguous slice of the key tiles and writes partial (m, l, o) states.
  // Head pairs (kKindVarlenHeads): query tile i is head h + i over the same
  // 128 rows, both heads of one KV group; otherwise tile i covers rows
  // [row0 + 128 i, row0 + 128 i + 128) of head h.
  constexpr bool HP =
      KIND == kKindVarlenHeads || KIND == kKindDenseHeads || KIND == kKindPagedHeads;
  constexpr bool PAGED = KIND == kKindPaged || KIND == kKindPagedHeads;  // K/V through a block table
  constexpr bool DENSE = KIND == kKindDense || KIND == kKindDenseHeads;  // [B, N, H, d] rows
  static_assert(!HP || QT == 2, "head pairs hold two query tiles");
  constexpr int kCtaRows = HP ? kPrefillBM : Sh::kRows;  // query rows per work item
  constexpr int kHeadStep = HP ? 2 : 1;                   // heads per work item
  const int split = (KIND == kKindDenseSplit) ? static_cast<int>(blockIdx.x % p.num_splits) : 0;
  const int lin = (KIND == kKindDenseSplit) ? static_cast<int>(blockIdx.x / p.num_splits)
                                            : static_cast<int>(blockIdx.x);
  // (unit, pair, h) of work item x; false past the last item.  Collective
  // over the warp for a compact packed batch.
  auto decode_item = [&](int x, int &unit_x, int &pair_x, int &h_x) -> bool {
    if ((KIND == kKindVarlen || KIND == kKindVarlenHeads) && p.compact)
      return varlen_compact_item<kCtaRows, kHeadStep>(p, x, CAUSAL, unit_x, pair_x, h_x);
    const int hgs = p.head_group / kHeadStep;  // head slots per ordering group
    const int slots = p.H / kHeadStep;
    const int h_in = x % hgs;
    const int t_lin = x / hgs;
    const int pair_rank = t_lin % p.max_pairs;
    const int grp = t_lin / p.max_pairs;
    h_x = ((grp % (slots / hgs)) * hgs + h_in) * kHeadStep;
    unit_x = grp / (slots / hgs);
    pair_x = CAUSAL ? (p.max_pairs - 1 - pair_rank) : pair_rank;
    return true;
  };
  int h, unit, pair;  // unit: batch element or sequence
  if (!decode_item(lin, unit, pair, h)) return;  // past the last item
  // len: query rows of the unit; kv_len: its keys; offset = kv_len - len
  // aligns causal masking to the bottom right (query i sees keys
  // j <= i + offset).
  int b, seq_start, len, kv_len, offset;
  if (DENSE || KIND == kKindDenseSplit) {
    b = unit;
    seq_start = 0;
    len = p.N;
    kv_len = len;
    offset = 0;
  } else {
    seq_start = checked_load(p.cu_seqlens, unit, p.B + 1, p.status);
    const int seq_end = checked_load(p.cu_seqlens, unit + 1, p.B + 1, p.status);
    if (seq_start < 0 || seq_end < seq_start || seq_end > p.total_tokens) {
      if (pair == 0 && h == 0) raise_status(p.status, FA_DEV_BAD_SEQLEN);
      return;
    }
    len = seq_end - seq_start;
    // Longer than max_seqlen: a grid sized from it cannot cover the sequence.
    // Any item of head 0 reports it; the sequence's first item, which is one,
    // is launched whenever the sequences before it respect max_seqlen.
    if (len > p.max_pairs * kCtaRows && h == 0) raise_status(p.status, FA_DEV_BAD_SEQLEN);
    b = 0;
    if (KIND == kKindVarlen || KIND == kKindVarlenHeads) {
      kv_len = len;
      offset = 0;
    } else {
      kv_len = checked_load(p.ctx_lens, unit, p.B, p.status);
      if (kv_len < 0 || kv_len > p.max_ctx_len ||
          kv_len > p.max_blocks_per_seq * kDecodeBlock) {
        if (pair == 0 && h == 0) raise_status(p.status, FA_DEV_BAD_CTX);
        return;
      }
      offset = kv_len - len;
    }
  }
  const int row0 = pair * kCtaRows;
  if (row0 >= len) return;  // no padding work: the whole CTA leaves before any set-up
  // first query row (within the sequence) and head of query tile i
  auto tile_row = [&](int i) { return HP ? row0 : row0 + i * kPrefillBM; };
  auto tile_head = [&](int i) { return HP ? h + i : h; };

  const int n_kv_all = (kv_len + kPrefillBN - 1) / kPrefillBN;
  int kv_end[kPrefillQTiles];
#pragma unroll
  for (int i = 0; i < kPrefillQTiles; ++i) {
    const int t0 = tile_row(i);
    if (i >= QT || t0 >= len) {
      kv_end[i] = 0;
    } else {
      int e = n_kv_all;
      if (CAUSAL) {
        const int last_key = min(t0 + kPrefillBM - 1, len - 1) + offset;
        e = (last_key < 0) ? 0 : min(n_kv_all, last_key / kPrefillBN + 1);
      }
      // a live tile runs at least one key tile (possibly fully masked), so
      // that rows which see no key are still written (O = 0, LSE = -inf)
      kv_end[i] = max(e, 1);
    }
  }
  // This CTA's key tiles are [kv0, kv0 + n_kv); from here on kv_end[i] counts
  // the tiles of query tile i inside that range.
  int kv0 = 0;
  if (KIND == kKindDenseSplit) {
    const int total = max(kv_end[0], kv_end[1]);
    const int per = (total + p.num_splits - 1) / p.num_splits;
    kv0 = split * per;
    const int stop = min(total, kv0 + per);
#pragma unroll
    for (int i = 0; i < kPrefillQTiles; ++i) kv_end[i] = max(0, min(kv_end[i], stop) - kv0);
  }
  const int n_kv = max(kv_end[0], kv_end[1]);
  const bool live1 = QT == 2 && tile_row(1) < len;  // the second query tile has rows

  // ---------------------------------------------------------- shared memory
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + SK;
  uint64_t *v_full = k_empty + SK;
  uint64_t *s_full = v_full + SV;
  uint64_t *p_full = s_full + 2;
  uint64_t *o_done = p_full + 2;
  uint64_t *drain = o_done + 2;
  uint64_t *v_empty = drain + 1;  // V-stage releases
  constexpr bool ONES = L::kOnes;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t *sQ = smem + L::kQ;
  uint8_t *sK = smem + L::kK;
  uint8_t *sV = smem + L::kV;
  const int kvh = h / p.group;
  // Dense kinds: K(0) is copied with Q, before the block-wide set-up ends.
  const bool k0_early = !PAGED && n_kv > 0;

  if (warp == Sh::kTmaWarp && lane == 0) {
    // The producer thread initialises the barriers and starts the Q copies
    // (and K(0)) right away; the other warps wait for it at __syncthreads.
    mbar_init(q_full, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < SV; ++s) mbar_init(&v_empty[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (PAGED) tma_prefetch_desc(&tm_v1);
    const int nq = live1 ? 2 : 1;
    mbar_arrive_expect_tx(q_full, nq * L::kTileBytes);
    for (int i = 0; i < nq; ++i) {
      const int qrow = seq_start + tile_row(i);
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_4d(sQ + i * L::kTileBytes + c * L::kChunkBytes, &tm_q, q_full,
                    c * L::kChunkElems, tile_head(i), qrow, b);
    }
    if (k0_early) {
      mbar_arrive_expect_tx(&k_full[0], L::kTileBytes);
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_4d(sK + c * L::kChunkBytes, &tm_k, &k_full[0], c * L::kChunkElems, kvh,
                    seq_start + kv0 * kPrefillBN, b);
    }
  }
  if (warp == Sh::kMmaWarp) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  if (PAGED) {
    // Rows of a V stage that no load fills (keys past the context in the last
    // key tile) must hold finite values: P is 0 there, but 0 * NaN is NaN.
    uint4 *z = reinterpret_cast<uint4 *>(smem + L::kV);
    for (int t = threadIdx.x; t < SV * L::kTileBytes / 16; t += Sh::kThreads)
      z[t] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (ONES) {
    // the block of ones read beside every V tile (bf16 1.0 = 0x3F80); the
    // 128-byte swizzle permutes equal values, so no pattern is needed
    uint4 *o1 = reinterpret_cast<uint4 *>(smem + L::kOnesOff);
    for (int t = threadIdx.x; t < L::kChunkBytes / 16; t += Sh::kThreads)
      o1[t] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  }
  if (PAGED || ONES) fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= Sh::kSoftmaxWarps) {
  // One query tile per CTA: this warpgroup (MMA, TMA, two idle warps) hands
  // registers to the softmax warpgroup.
  if constexpr (QT == 1) setmaxnreg_dec<kPrefill1CtlRegs>();
  const bool k_producer = warp == Sh::kTmaWarp;  // else the V producer
  if ((warp == Sh::kTmaWarp || warp == Sh::kTmaVWarp) && PAGED) {
    // ------------------------------------------------------ TMA producer, paged
    // The warp runs converged: lanes 0..7 look up the 8 physical blocks of a
    // 128-key tile in the block table, lane 0 issues the copies.  A block
    // whose id is outside the pool is not loaded (its keys hold stale data,
    // the status word records the error).  In the last block only the slots
    // inside the context are copied (one-row boxes for V), so stale slots of
    // the pool never reach shared memory.
    const int32_t *trow = p.block_table + static_cast<size_t>(unit) * p.max_blocks_per_seq;
    constexpr int kBlkPerTile = kPrefillBN / kDecodeBlock;
    constexpr uint32_t kRowBytes = 128 * L::kChunks;  // one key row, all chunks
    const int total_blk = (kv_len + kDecodeBlock - 1) / kDecodeBlock;
    int k_issued = 0, v_issued = 0;
    // The block table is read ahead: one coalesced load brings the 32 block
    // ids of 4 consecutive key tiles (lane = 8 * tile + slot), fetched 4
    // tiles before they are needed, so no copy waits on a table lookup.
    // Ids of tiles outside this CTA's range, or past the context, are -1;
    // an id outside the pool is reported and not loaded.
    auto fetch = [&](int w) -> int {
      const int blk = (kv0 + w) * kBlkPerTile + lane;
      if (w + lane / kBlkPerTile >= n_kv || blk >= total_blk) return -1;
      if (!in_bounds(static_cast<size_t>(trow - p.block_table) + blk, 1,
                     static_cast<size_t>(p.B) * p.max_blocks_per_seq, p.status))
        return -1;
      const int phys = trow[blk];
      if (phys < 0 || phys >= p.num_blocks) {
        raise_status(p.status, FA_DEV_BAD_BLOCK);
        return -1;
      }
      return phys;
    };
    constexpr int kWin = 32 / kBlkPerTile;
    int win_cur = fetch(0), win_nxt = fetch(kWin), win_base = 0;
    // physical block of slot `lane` of tile j (or -1), and its valid rows;
    // tiles are looked up in increasing order
    auto lookup = [&](int j, int &rows) -> int {
      if (j >= win_base + kWin) {
        win_base += kWin;
        win_cur = win_nxt;
        win_nxt = fetch(win_base + kWin);
      }
      const int phys = __shfl_sync(0xffffffffu, win_cur, ((j - win_base) * kBlkPerTile + lane) & 31);
      const int blk = (kv0 + j) * kBlkPerTile + lane;
      rows = 0;
      if (lane >= kBlkPerTile || phys < 0) return -1;
      rows = min(kDecodeBlock, kv_len - blk * kDecodeBlock);
      return phys;
    };
    // One copy per (block, 64-column chunk); the lanes issue them together
    // (lane = slot * kChunks + chunk), after lane 0 has posted the byte count.
    constexpr int kCopyLanes = kBlkPerTile * L::kChunks;
    const int my_t = lane / L::kChunks, my_c = lane % L::kChunks;
    auto load_k = [&](int j) -> bool {
      const int sk = j % SK;
      if (j >= SK && !mbar_wait_warp(&k_empty[sk], ((j / SK) - 1) & 1, abort_flag, p.status))
        return false;
      int rows;
      const int phys = lookup(j, rows);
      const uint32_t bytes =
          __reduce_add_sync(0xffffffffu, phys >= 0 ? kDecodeBlock * kRowBytes : 0u);
      if (lane == 0) mbar_arrive_expect_tx(&k_full[sk], bytes);
      __syncwarp();
      const int pb = __shfl_sync(0xffffffffu, phys, my_t & 7);
      if (lane < kCopyLanes && pb >= 0)
        tma_load_3d(sK + sk * L::kTileBytes + my_c * L::kChunkBytes + my_t * kDecodeBlock * 128,
                    &tm_k, &k_full[sk], my_c * L::kChunkElems, kvh, pb * kDecodeBlock);
      k_issued = j + 1;
      return true;
    };
    auto load_v = [&](int j) -> bool {
      const int sv = j % SV;
      if (j >= SV && !mbar_wait_warp(&v_empty[sv], ((j / SV) - 1) & 1, abort_flag, p.status))
        return false;
      int rows;
      const int phys = lookup(j, rows);
      const uint32_t bytes =
          __reduce_add_sync(0xffffffffu, phys >= 0 ? static_cast<uint32_t>(rows) * kRowBytes : 0u);
      if (lane == 0) mbar_arrive_expect_tx(&v_full[sv], bytes);
      __syncwarp();
      uint8_t *stage = sV + sv * L::kTileBytes;
      // whole blocks
      const int pb = __shfl_sync(0xffffffffu, phys, my_t & 7);
      const int nr = __shfl_sync(0xffffffffu, rows, my_t & 7);
      if (lane < kCopyLanes && pb >= 0 && nr == kDecodeBlock)
        tma_load_3d(stage + my_c * L::kChunkBytes + my_t * kDecodeBlock * 128, &tm_v, &v_full[sv],
                    my_c * L::kChunkElems, kvh, pb * kDecodeBlock);
      // the block holding the end of the context: only its rows inside the
      // context, one row per copy (lane = row * kChunks + chunk)
      const unsigned part =
          __ballot_sync(0xffffffffu, lane < kBlkPerTile && phys >= 0 && rows < kDecodeBlock);
      if (part != 0u) {
        const int tp = __ffs(part) - 1;
        const int pbp = __shfl_sync(0xffffffffu, phys, tp);
        const int nrp = __shfl_sync(0xffffffffu, rows, tp);
        const int rr = lane / L::kChunks;
        if (rr < nrp)
          tma_load_3d(stage + my_c * L::kChunkBytes + (tp * kDecodeBlock + rr) * 128, &tm_v1,
                      &v_full[sv], my_c * L::kChunkElems, kvh, pbp * kDecodeBlock + rr);
      }
      v_issued = j + 1;
      return true;
    };
    for (int j = 0; j < n_kv; ++j)
      if (!(k_producer ? load_k(j) : load_v(j))) break;
    if (lane == 0) {
      if (k_producer) {
        mbar_drain(q_full, 0, p.status);
        for (int j = max(0, k_issued - SK); j < k_issued; ++j)
          mbar_drain(&k_full[j % SK], (j / SK) & 1, p.status);
      } else {
        for (int j = max(0, v_issued - SV); j < v_issued; ++j)
          mbar_drain(&v_full[j % SV], (j / SV) & 1, p.status);
      }
    }
  } else if (warp == Sh::kTmaWarp) {
    // ------------------------------------------------------ TMA producer
    // The Q tiles of the work item that starts about a wave after this one
    // are read from HBM once: prefetch them into L2 now, so that CTA's first
    // S waits for L2 instead of HBM.
    if (KIND != kKindDenseSplit && p.prefetch_ahead > 0) {
      const long long ahead = static_cast<long long>(lin) + p.prefetch_ahead;
      int unit2 = 0, pair2 = 0, h2 = 0;
      if (ahead < static_cast<long long>(gridDim.x) &&
          decode_item(static_cast<int>(ahead), unit2, pair2, h2)) {
        int start2 = 0, len2 = p.N;
        if (!DENSE) {
          start2 = checked_load(p.cu_seqlens, unit2, p.B + 1, p.status);
          len2 = min(checked_load(p.cu_seqlens, unit2 + 1, p.B + 1, p.status), p.total_tokens) -
                 start2;
        }
        const int r2 = pair2 * kCtaRows;
        if (lane == 0 && start2 >= 0 && r2 < len2) {
          for (int i = 0; i < QT; ++i) {
            const int t2 = HP ? r2 : r2 + i * kPrefillBM;
            if (t2 >= len2) break;
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
              tma_prefetch_4d(&tm_q, c * L::kChunkElems, HP ? h2 + i : h2, start2 + t2,
                              DENSE ? unit2 : 0);
          }
        }
      }
    }
    if (lane == 0) {
      // Issue order K(0) (already issued with Q), then V(j), K(j+1) for
      // every j: a V load never waits behind a K stage that frees later.
      int k_issued = k0_early ? 1 : 0, v_issued = 0;
      auto load_k = [&](int j) -> bool {
        const int sk = j % SK;
        if (j >= SK && !mbar_wait(&k_empty[sk], ((j / SK) - 1) & 1, abort_flag, p.status))
          return false;
        mbar_arrive_expect_tx(&k_full[sk], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sK + sk * L::kTileBytes + c * L::kChunkBytes, &tm_k, &k_full[sk], c * L::kChunkElems,
                      kvh, seq_start + (kv0 + j) * kPrefillBN, b);
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int sv = j % SV;
        if (j >= SV && !mbar_wait(&v_empty[sv], ((j / SV) - 1) & 1, abort_flag, p.status))
          return false;
        mbar_arrive_expect_tx(&v_full[sv], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sV + sv * L::kTileBytes + c * L::kChunkBytes, &tm_v, &v_full[sv], c * L::kChunkElems,
                      kvh, seq_start + (kv0 + j) * kPrefillBN, b);
        v_issued = j + 1;
        return true;
      };
      if (n_kv > 0 && (k0_early || load_k(0))) {
        for (int j = 0; j < n_kv; ++j) {
          if (!load_v(j)) break;
          if (j + 1 < n_kv && !load_k(j + 1)) break;
        }
      }
      // Never leave copies in flight into shared memory that is about to be
      // released: wait for the last load of every stage.
      mbar_drain(q_full, 0, p.status);
      for (int j = max(0, k_issued - SK); j < k_issued; ++j)
        mbar_drain(&k_full[j % SK], (j / SK) & 1, p.status);
      for (int j = max(0, v_issued - SV); j < v_issued; ++j)
        mbar_drain(&v_full[j % SV], (j / SV) & 1, p.status);
    }
  } else if (warp == Sh::kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged; elect.sync picks the lane
    // that issues each tcgen05 instruction.
    {
      // one MMA consumes 32 bytes of the contraction: 16 bf16 or 32 e4m3 values
      constexpr int kKStep = 32 / L::kElemBytes;
      constexpr uint32_t kIdescS = FP8 ? idesc_e4m3_f32(kPrefillBM, kPrefillBN, false, false)
                                       : idesc_bf16_f32(kPrefillBM, kPrefillBN, false, false);
      constexpr uint32_t kIdescO = FP8 ? idesc_e4m3_f32(kPrefillBM, D, false, true)
                                       : idesc_bf16_f32(kPrefillBM, L::kOCols, false, true);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t k_base = smem_u32(sK);
      const uint32_t v_base = smem_u32(sV);

      // One lane (the same one every time: the warp is converged) issues a
      // whole product and its commit; the K-steps advance the descriptors'
      // address fields (address / 16) by constants.
      auto issue_s = [&](int i, int st) {
        const uint32_t d_t = tmem + i * 128;
        if (elect_one()) {
          const uint64_t a0 = sdesc_swz<L::kSwz>(q_base + i * L::kTileBytes, 16, L::kSbo);
          const uint64_t b0 = sdesc_swz<L::kSwz>(k_base + st * L::kTileBytes, 16, L::kSbo);
          constexpr int kStepsPerRow = L::kSwz / 32;  // 32-byte K-steps in a swizzled row
#pragma unroll
          for (int kk = 0; kk < D / kKStep; ++kk) {
            const uint64_t off = static_cast<uint64_t>(
                ((kk / kStepsPerRow) * L::kChunkBytes + (kk % kStepsPerRow) * 32) >> 4);
            if (FP8)
              mma_ss_f8(d_t, a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
            else
              mma_ss(d_t, a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[i]);
        }
        __syncwarp();
      };
      auto issue_o = [&](int i, int st, int j) {
        const uint32_t d_t = tmem + L::kTmemO + i * L::kOCols;
        const uint32_t p_t = tmem + i * 128;
        if (elect_one()) {
          // N beyond D (the ones block) is read at the leading-byte offset
          const uint32_t lbo = ONES ? static_cast<uint32_t>(L::kOnesOff - (L::kV + st * L::kTileBytes))
                                    : static_cast<uint32_t>(L::kChunkBytes);
          const uint64_t b0 = sdesc_swz<L::kSwz>(v_base + st * L::kTileBytes, lbo, L::kSbo);
#pragma unroll
          for (int kk = 0; kk < kPrefillBN / kKStep; ++kk) {
            // kKStep keys of swizzled rows; P holds kKStep keys in 8 TMEM columns
            const uint64_t off = static_cast<uint64_t>((kk * kKStep * L::kSwz) >> 4);
            if (FP8)
              mma_ts_f8(d_t, p_t + kk * 8, b0 + off, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
            else
              mma_ts(d_t, p_t + kk * 8, b0 + off, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
          }
          // only the epilogue waits for O (the O rescale in the softmax is
          // ordered by the S commit, which covers every earlier product)
          if (j == kv_end[i] - 1) mma_commit(&o_done[i]);
        }
        __syncwarp();
      };

      // Issue order per key tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
      // that each softmax warpgroup works while the tensor pipe runs the
      // other tile's products.  S_i(j+1) reuses the TMEM columns that PV_i(j),
      // issued just before it by this thread, reads P_i(j) from; tcgen05 MMAs
      // issued by one thread execute in order.
      // (a split that owns no key tile issues nothing)
      bool ok = n_kv > 0 && mbar_wait_warp(q_full, 0, abort_flag, p.status) &&
                mbar_wait_warp(&k_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < 2; ++i)
          if (kv_end[i] > 0) issue_s(i, 0);
        mma_commit_elect(&k_empty[0]);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int sv = j % SV;
        const int sk1 = (j + 1) % SK;
        bool k_next = false;
        auto wait_k_next = [&]() -> bool {
          if (k_next) return true;
          if (!mbar_wait_warp(&k_full[sk1], ((j + 1) / SK) & 1, abort_flag, p.status)) return false;
          tc_fence_after();
          k_next = true;
          return true;
        };
        // With dense K/V, V(j) and K(j+1) are usually resident before P_0(j)
        // is ready: waiting for them first keeps both waits off the path
        // from P_i(j) to S_i(j+1).  (Their loads never depend on this
        // iteration's releases, so the order cannot deadlock.)  Gathered
        // paged K may still be in flight, so that kind waits for K(j+1)
        // only before the S MMAs that read it.
        if (!mbar_wait_warp(&v_full[sv], (j / SV) & 1, abort_flag, p.status)) break;
        if (!PAGED && SK > 1 && j + 1 < n_kv && !wait_k_next()) break;
        tc_fence_after();
        if (j < kv_end[0]) {
          if (!mbar_wait_warp(&p_full[0], j & 1, abort_flag, p.status)) break;
          tc_fence_after();
          issue_o(0, sv, j);
        }
        if (j + 1 < kv_end[0]) {
          if (!wait_k_next()) break;
          issue_s(0, sk1);
        }
        if (j < kv_end[1]) {
          if (!mbar_wait_warp(&p_full[1], j & 1, abort_flag, p.status)) break;
          tc_fence_after();
          issue_o(1, sv, j);
        }
        // the V stage of key tile j is free once its P V products are done
        mma_commit_elect(&v_empty[sv]);
        if (j + 1 < kv_end[1]) {
          if (!wait_k_next()) break;
          issue_s(1, sk1);
        }
        // the stage of K(j+1) is free once S_0(j+1) and S_1(j+1) are done
        if (j + 1 < n_kv) mma_commit_elect(&k_empty[sk1]);
      }
      // Everything this thread issued must finish before TMEM is released.
      mma_commit_elect(drain);
      mbar_drain(drain, 0, p.status);
    }
  }
  } else {
    if constexpr (QT == 1) setmaxnreg_inc<kPrefill1SoftmaxRegs>();
    // ------------------------------------------------------ softmax warpgroups
    const int i = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + i * 128 + lane_off;
    const uint32_t tO = tmem + L::kTmemO + i * L::kOCols + lane_off;
    const int qi = tile_row(i) + row;  // query row within the sequence
    const int hi = tile_head(i);       // query head of this tile
    const int my_end = kv_end[i];
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    // Reference maximum of the exponentials, log2 units.  It follows the row
    // maximum, but moves only when the maximum grows by more than
    // kRescaleLog2: until then every p stays below 2^kRescaleLog2, which the
    // fp32 sum and the bf16 P operand hold as well as values below 1.  o and
    // l always share the reference, so o / l is the same result; O in TMEM
    // is rescaled only when the reference moves.
    float m_ref = -CUDART_INF_F;
    float l = 0.f;        // running sum of the bf16 P values, relative to m_ref
    float l_exact = 0.f;  // running sum of the fp32 exponentials, relative to m_ref
    bool ok = true;
    // keys [0, limit) are visible to this row (bottom-right causal alignment)
    const int limit = CAUSAL ? min(kv_len, qi + 1 + offset) : kv_len;

    for (int j = 0; j < my_end; ++j) {
      ok = mbar_wait(&s_full[i], j & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();

      uint32_t sr[128];
      tmem_ld128_wait(tS, sr);
      const int nvis = limit - (kv0 + j) * kPrefillBN;
      // keys past the last one any row of this warp sees (the causal
      // diagonal): at d = 64, where the softmax bounds the key loop, their
      // 64-key halves of P are zero without exponentials
      const int nvis_w = (D == 64) ? __reduce_max_sync(0xffffffffu, nvis) : kPrefillBN;
      if (__any_sync(0xffffffffu, nvis < kPrefillBN)) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= nvis) sr[c] = 0xff800000u;  // -inf
      }
      // four independent three-input max chains over the 128 scores
      auto f = [&](int c) { return __uint_as_float(sr[c]); };
      float mx0 = f(0), mx1 = f(1), mx2 = f(2), mx3 = f(3);
#pragma unroll
      for (int c = 4; c < 124; c += 8) {
        mx0 = fmax3(mx0, f(c), f(c + 1));
        mx1 = fmax3(mx1, f(c + 2), f(c + 3));
        mx2 = fmax3(mx2, f(c + 4), f(c + 5));
        mx3 = fmax3(mx3, f(c + 6), f(c + 7));
      }
      mx0 = fmax3(mx0, f(124), f(125));
      mx1 = fmax3(mx1, f(126), f(127));
      const float m_new = fmaxf(m_ref, fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2);
      // false while nothing visible has been seen (both -inf)
      const bool grow = m_new > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_ref - m_new);  // 0 on the first visible tile
        m_ref = m_new;
      }
      // NaN guard ("exp(-inf - -inf) is NaN"): a row that has seen no
      // visible key yet uses the finite reference 0, so every p is 0.
      const float m_use = (m_ref == -CUDART_INF_F) ? 0.f : m_ref;
      const float2 negm = make_float2(-m_use, -m_use);
      // Two row sums: l sums the bf16 values that the P V product multiplies,
      // so o / l is a weighted mean with consistent weights (with the ones
      // block, the tensor cores form it in column D of O); l_exact sums the
      // fp32 exponentials and gives the log-sum-exp.
      float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
      float2 re0 = make_float2(0.f, 0.f), re1 = make_float2(0.f, 0.f);
      // P in two halves of 64 keys, each stored to TMEM as soon as it is packed
      if (!FP8) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
          if (D == 64 && half * 64 >= nvis_w) {
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = 0u;
            tmem_st32(tS + half * 32, pk);
            continue;
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int e = half * 64 + 2 * c;
            const float2 x0 = ffma2(
                make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, negm);
            const float2 x1 = ffma2(
                make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2x2, negm);
            const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
            const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
            pk[c] = pack_bf16x2(p0.x, p0.y);
            pk[c + 1] = pack_bf16x2(p1.x, p1.y);
            re0 = fadd2(re0, p0);
            re1 = fadd2(re1, p1);
            if (!ONES) {
              add_bf16x2_to(rs0, pk[c]);
              add_bf16x2_to(rs1, pk[c + 1]);
            }
          }
          tmem_st32(tS + half * 32, pk);
        }
      } else {
        // e4m3 P, four keys per TMEM column.  Its 3-bit mantissa leaves the
        // weights as they are rounded; both sums use the fp32 exponentials.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int e = half * 64 + 4 * c;
            const float2 x0 = ffma2(
                make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, negm);
            const float2 x1 = ffma2(
                make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2x2, negm);
            const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
            const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
            pk[c] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
            re0 = fadd2(re0, p0);
            re1 = fadd2(re1, p1);
          }
          tmem_st16(tS + half * 16, pk);
        }
        rs0 = re0;
        rs1 = re1;
      }
      const float2 rs = fadd2(rs0, rs1);
      const float2 re = fadd2(re0, re1);
      if (!ONES) l = l * alpha + (rs.x + rs.y);
      l_exact = l_exact * alpha + (re.x + re.y);
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + c * 32, o);
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            const float2 v = fmul2(make_float2(__uint_as_float(o[t]), __uint_as_float(o[t + 1])), a2);
            o[t] = __float_as_uint(v.x);
            o[t + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tO + c * 32, o);
        }
        if (ONES) {  // the row-sum columns follow O
          uint32_t o[16];
          tmem_ld16_wait(tO + D, o);
#pragma unroll
          for (int t = 0; t < 16; t += 2) {
            const float2 v = fmul2(make_float2(__uint_as_float(o[t]), __uint_as_float(o[t + 1])), a2);
            o[t] = __float_as_uint(v.x);
            o[t + 1] = __float_as_uint(v.y);
          }
          tmem_st16(tO + D, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[i]);
    }
    const float m = m_ref;

    // ---------------------------------------------------- epilogue
    if constexpr (KIND == kKindDenseSplit) {
      // Partial state of this split: o unnormalised (fp32), m (log2 units),
      // l over the bf16 weights and l over the fp32 exponentials.  A row of
      // a live tile that got no key tile stores the neutral state.
      const bool tile_live = row0 + i * kPrefillBM < len;
      bool have = ok && my_end > 0;
      if (have) {
        have = mbar_wait(&o_done[i], 0, abort_flag, p.status);
        have = __all_sync(0xffffffffu, have);
      }
      if (ONES && have) {  // the sum of the bf16 weights, from column D of O
        tc_fence_after();
        uint32_t lr[16];
        tmem_ld16_wait(tO + D, lr);
        l = __uint_as_float(lr[0]);
      }
      if (tile_live && my_end > 0) {
        // The fp32 tile goes out through the warpgroup's free Q tile (it
        // holds half of an fp32 tile), half of the columns at a time, with
        // one TMA store per 32-column chunk of 128-byte swizzled rows; rows
        // past N are clipped by the tensor bounds.  All four warps meet at
        // the barriers (the conditions above are the same for the whole
        // tile); a warp whose wait gave up writes nothing, and the status
        // word already marks the call as failed.
        if (have) tc_fence_after();
        uint8_t *stile = sQ + i * L::kTileBytes;
        constexpr int kHalfChunks = D / 64;
        static_assert(kHalfChunks * L::kChunkBytes <= L::kTileBytes, "staging tile too small");
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int cc = 0; have && cc < kHalfChunks; ++cc) {
            const int c = half * kHalfChunks + cc;  // columns [32 c, 32 c + 32)
            uint32_t o[32];
            tmem_ld32_wait(tO + c * 32, o);
            uint8_t *srow = stile + cc * L::kChunkBytes + row * 128;
            // 128-byte swizzle: 16-byte unit u of row r sits at u ^ (r % 8)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4 *>(srow + ((u ^ (row & 7)) * 16)) =
                  make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + i, 128);
          if (row == 0 && have) {
#pragma unroll
            for (int cc = 0; cc < kHalfChunks; ++cc)
              tma_store_4d(&tm_o, stile + cc * L::kChunkBytes, (half * kHalfChunks + cc) * 32,
                           h, row0 + i * kPrefillBM, split * p.B + b);
            tma_store_commit();
            tma_store_wait_read();
          }
          // the second half reuses the staging tile once the copies have read it
          if (half == 0) named_bar_sync(1 + i, 128);
        }
      }
      if (tile_live && (have || my_end == 0) && qi < len) {
        const size_t prow = (static_cast<size_t>(split) * p.B + b) * p.N + qi;
        if (in_bounds(prow * p.H + h, 1,
                      static_cast<size_t>(p.num_splits) * p.B * p.N * p.H, p.status))
          reinterpret_cast<float4 *>(p.ml_part)[prow * p.H + h] =
            have ? make_float4(m, l, l_exact, 0.f) : make_float4(-CUDART_INF_F, 0.f, 0.f, 0.f);
      }
    } else if (my_end > 0) {
      if (ok) {
        ok = mbar_wait(&o_done[i], 0, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
      }
      {
        if (ok) tc_fence_after();
        if (ONES && ok) {  // the sum of the bf16 weights, from column D of O
          uint32_t lr[16];
          tmem_ld16_wait(tO + D, lr);
          l = __uint_as_float(lr[0]);
        }
        const bool live = qi < len;
        const float inv_l = (l > 0.f) ? p.v_descale / l : 0.f;
        // A whole bf16 tile goes out through shared memory and one TMA store
        // per 64-column chunk (rows past the end of a dense sequence are
        // clipped by the tensor bounds).  The warpgroup's Q tile is free: its
        // last S MMA completed before the last S tile was handed over.  An
        // fp8 Q tile holds half of the bf16 output tile at d = 128, so the
        // tile leaves in two passes of 64 columns; at d = 64 (a quarter) and
        // for a partial tile of a packed layout, whose tail rows belong to
        // the next sequence, the rows are written one by one instead.
        constexpr int kOutChunkBytes = 128 * 128;  // 128 rows x 64 bf16 columns
        constexpr int kPasses = FP8 ? 2 : 1;
        constexpr int kPassCols = D / 32 / kPasses;  // 32-column TMEM chunks per pass
        const bool tma_out =
            (!FP8 || D == 128) && (DENSE || tile_row(i) + kPrefillBM <= len);
        if (tma_out) {
          // All four warps of the tile meet at the barriers below (my_end and
          // tma_out are the same for the whole tile); a warp whose wait gave
          // up writes nothing, and the status word already marks the call as
          // failed.
          uint8_t *stile = sQ + i * L::kTileBytes;
          static_assert(kPassCols / 2 * kOutChunkBytes <= L::kTileBytes, "output staging tile");
#pragma unroll
          for (int pass = 0; pass < kPasses; ++pass) {
#pragma unroll
          for (int cc = 0; ok && cc < kPassCols; ++cc) {
            const int c = pass * kPassCols + cc;
            uint32_t o[32];
            tmem_ld32_wait(tO + c * 32, o);
            uint8_t *srow = stile + (cc >> 1) * kOutChunkBytes + row * 128;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[v4 * 8 + 0]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(o[v4 * 8 + 2]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(o[v4 * 8 + 4]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(o[v4 * 8 + 6]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 7]) * inv_l);
              // 128-byte swizzle: 16-byte unit u of row r sits at u ^ (r % 8)
              const int u = ((c & 1) * 4 + v4) ^ (row & 7);
              *reinterpret_cast<uint4 *>(srow + u * 16) = w;
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + i, 128);
          if (row == 0 && ok) {
            const int orow = (DENSE ? 0 : seq_start) + tile_row(i);
#pragma unroll
            for (int c = 0; c < kPassCols / 2; ++c)
              tma_store_4d(&tm_o, stile + c * kOutChunkBytes, (pass * kPassCols / 2 + c) * 64, hi,
                           orow, b);
            tma_store_commit();
            tma_store_wait_read();
          }
          // the next pass reuses the staging tile once the copies have read it
          if (pass + 1 < kPasses) named_bar_sync(1 + i, 128);
          }
        }
        size_t out_row;
        if (!DENSE)
          out_row = static_cast<size_t>(seq_start + qi);
        else
          out_row = static_cast<size_t>(b) * p.N + qi;
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) +
                                               ((out_row * p.H + hi) * D) * 2);
        // rows of the output (and of the log-sum-exp) the call owns
        const size_t out_rows =
            DENSE ? static_cast<size_t>(p.B) * p.N : static_cast<size_t>(p.total_tokens);
        const bool row_ok =
            !live || tma_out || in_bounds((out_row * p.H + hi) * D, D, out_rows * p.H * D, p.status);
#pragma unroll
        for (int c = 0; ok && !tma_out && c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + c * 32, o);  // warp-wide: every lane loads
          if (live && row_ok) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[v4 * 8 + 0]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(o[v4 * 8 + 2]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(o[v4 * 8 + 4]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(o[v4 * 8 + 6]) * inv_l,
                                __uint_as_float(o[v4 * 8 + 7]) * inv_l);
              dst[c * 4 + v4] = w;
            }
          }
        }
        const size_t lse_idx = !DENSE
                                   ? static_cast<size_t>(hi) * p.total_tokens + seq_start + qi
                                   : (static_cast<size_t>(b) * p.H + hi) * p.N + qi;
        if (ok && live && p.lse != nullptr && in_bounds(lse_idx, 1, out_rows * p.H, p.status)) {
          p.lse[lse_idx] = (l_exact > 0.f) ? (m + __log2f(l_exact)) * 0.69314718055994530942f
                                           : -CUDART_INF_F;
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == Sh::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ------------------------------------------------------------------ split combine
// One warp per (batch, row, head) merges the partial states of the splits
// with the rescaling of the explainer page's "Show the maths":
// M = max m_s, o = sum 2^(m_s - M) o_s / sum 2^(m_s - M) l_s,
// lse = (M + log2 sum 2^(m_s - M) l_exact_s) ln 2.
template <int D>
__global__ void __launch_bounds__(128) prefill_split_combine_kernel(const PrefillParams p) {
  pdl_wait_primary();  // the split grid's partial states are complete from here on
  // The split grid has raised all its status bits: one thread reads them
  // here and publishes them as the call's status when its row is done.
  const bool publisher = blockIdx.x == 0 && threadIdx.x == 0 && p.call != nullptr;
  const unsigned int call_bits = publisher ? call_status_bits(p.call) : 0u;
  // this kernel's own (checked-build) index errors go to the device word only
  unsigned int *status = p.call != nullptr ? p.dev_status : p.status;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const size_t rows = static_cast<size_t>(p.B) * p.N * p.H;
  const size_t gw = static_cast<size_t>(blockIdx.x) * 4 + warp;
  if (gw >= rows) return;
  const size_t bn = gw / p.H;  // b * N + n
  const int h = static_cast<int>(gw % p.H);
  const size_t stride = static_cast<size_t>(p.B) * p.N * p.H;  // between splits
  const size_t parts = static_cast<size_t>(p.num_splits) * stride;  // partial rows
  // (m, l, l_exact) of split s for this row (the neutral state if the index
  // fails a check of the checked build)
  auto ml = [&](int sp) -> float4 {
    const size_t idx = sp * stride + gw;
    return in_bounds(idx, 1, parts, status) ? reinterpret_cast<const float4 *>(p.ml_part)[idx]
                                              : make_float4(-CUDART_INF_F, 0.f, 0.f, 0.f);
  };
  // M = max over the splits, one split per lane (at most 16 splits)
  float M = (lane < p.num_splits) ? ml(lane).x : -CUDART_INF_F;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float Ls = 0.f, Le = 0.f;
  // Split s adds 2^(m_s - M) (l_s, l_exact_s, o_s), four splits per memory
  // round trip; a split without keys for this row (m_s = -inf) is passed
  // over by a select, so its o_s slot never reaches the output.
  if (M != -CUDART_INF_F) {
    auto add = [&](const float4 st, const float (&v)[E]) {
      const bool live = st.x != -CUDART_INF_F;
      const float w = ex2(st.x - M);
      Ls = live ? fmaf(w, st.y, Ls) : Ls;
      Le = live ? fmaf(w, st.z, Le) : Le;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = live ? fmaf(w, v[e], acc[e]) : acc[e];
    };
    auto load_o = [&](int sp, float (&v)[E]) {
      const size_t idx = (sp * stride + gw) * D + lane * E;
      const bool in = in_bounds(idx, E, parts * D, status);
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = in ? p.o_part[idx + e] : 0.f;
    };
    constexpr int U = 4;
    int sp = 0;
    for (; sp + U <= p.num_splits; sp += U) {
      float4 st[U];
      float v[U][E];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        st[u] = ml(sp + u);
        load_o(sp + u, v[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) add(st[u], v[u]);
    }
    for (; sp < p.num_splits; ++sp) {
      float v[E];
      load_o(sp, v);
      add(ml(sp), v);
    }
  }
  const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
  uint16_t *dst = static_cast<uint16_t *>(p.out) + gw * D + lane * E;
  if (in_bounds(gw * D + lane * E, E, rows * D, status)) {
#pragma unroll
    for (int e = 0; e < E; e += 2)
      *reinterpret_cast<uint32_t *>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  }
  const size_t b = bn / p.N, n = bn % p.N;
  const size_t lse_idx = (b * p.H + h) * p.N + n;
  if (lane == 0 && p.lse != nullptr && in_bounds(lse_idx, 1, rows, status))
    p.lse[lse_idx] = (Le > 0.f) ? (M + __log2f(Le)) * 0.69314718055994530942f : -CUDART_INF_F;
  if (publisher) publish_call_status(p.call, call_bits, p.dev_status);
}

cudaError_t launch_prefill_split_combine(const PrefillParams &p, int d, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(p.B) * p.N * p.H;
  // launched as a programmatic dependent of the split grid on the same stream
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (d == 64) return cudaLaunchKernelEx(&cfg, prefill_split_combine_kernel<64>, p);
  return cudaLaunchKernelEx(&cfg, prefill_split_combine_kernel<128>, p);
}

// Publishes the status of a split-KV call that ran the plain kernel alone
// (one split), once that kernel has completed.
__global__ void __launch_bounds__(32) call_status_kernel(CallStatus *call, unsigned int *dev) {
  if (threadIdx.x == 0) publish_call_status(call, call_status_bits(call), dev);
}

cudaError_t launch_call_status(CallStatus *call, unsigned int *dev, cudaStream_t stream) {
  call_status_kernel<<<1, 32, 0, stream>>>(call, dev);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ launch

template <int D, bool CAUSAL, int KIND, bool FP8 = false, int QT = 2>
static cudaError_t launch_prefill_t(const CUtensorMap &tq, const CUtensorMap &tk,
                                    const CUtensorMap &tv, const CUtensorMap &tv1,
                                    const CUtensorMap &to, const PrefillParams &p, int grid,
                                    cudaStream_t stream) {
  using L = PrefillLayout<D, FP8, QT>;
  using Sh = PrefillShape<QT>;
  auto kern = prefill_kernel<D, CAUSAL, KIND, FP8, QT>;
  if constexpr (QT == 1) {
    // The setmaxnreg split assumes kPrefill1LaunchRegs registers per thread
    // at launch; with fewer, the register increase could never be granted,
    // so such a build is refused instead of launched.
    static const int launch_regs = [&] {
      cudaFuncAttributes a{};
      return cudaFuncGetAttributes(&a, kern) == cudaSuccess ? a.numRegs : -1;
    }();
    if (launch_regs != kPrefill1LaunchRegs) return cudaErrorInvalidKernelImage;
  }
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, Sh::kThreads, L::kSmemAlloc, stream>>>(tq, tk, tv, tv1, to, p);
  return cudaGetLastError();
}

template <int D, int KIND, int QT = 2>
static cudaError_t launch_prefill_k(const CUtensorMap &tq, const CUtensorMap &tk,
                                    const CUtensorMap &tv, const CUtensorMap &tv1,
                                    const CUtensorMap &to, const PrefillParams &p, bool causal,
                                    int grid, cudaStream_t stream) {
  return causal ? launch_prefill_t<D, true, KIND, false, QT>(tq, tk, tv, tv1, to, p, grid, stream)
                : launch_prefill_t<D, false, KIND, false, QT>(tq, tk, tv, tv1, to, p, grid, stream);
}

// FP8 prefill, d = 64 or 128: dense batches and packed sequences (row pairs
// or head pairs); `to` is the bf16 output map (used at d = 128).
template <int D, int KIND>
static cudaError_t launch_prefill_fp8_k(const CUtensorMap &tq, const CUtensorMap &tk,
                                        const CUtensorMap &tv, const CUtensorMap &to,
                                        const PrefillParams &p, bool causal, int grid,
                                        cudaStream_t stream) {
  return causal ? launch_prefill_t<D, true, KIND, true>(tq, tk, tv, tv, to, p, grid, stream)
                : launch_prefill_t<D, false, KIND, true>(tq, tk, tv, tv, to, p, grid, stream);
}

template <int D>
static cudaError_t launch_prefill_fp8_d(const CUtensorMap &tq, const CUtensorMap &tk,
                                        const CUtensorMap &tv, const CUtensorMap &to,
                                        const PrefillParams &p, bool causal, int grid,
                                        cudaStream_t stream, int kind) {
  if (kind == kKindVarlen)
    return launch_prefill_fp8_k<D, kKindVarlen>(tq, tk, tv, to, p, causal, grid, stream);
  if (kind == kKindVarlenHeads)
    return launch_prefill_fp8_k<D, kKindVarlenHeads>(tq, tk, tv, to, p, causal, grid, stream);
  return launch_prefill_fp8_k<D, kKindDense>(tq, tk, tv, to, p, causal, grid, stream);
}

cudaError_t launch_prefill_fp8(const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, const CUtensorMap &to,
                               const PrefillParams &p, bool causal, int grid,
                               cudaStream_t stream, int kind, int d) {
  return d == 64 ? launch_prefill_fp8_d<64>(tq, tk, tv, to, p, causal, grid, stream, kind)
                 : launch_prefill_fp8_d<128>(tq, tk, tv, to, p, causal, grid, stream, kind);
}

cudaError_t launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const CUtensorMap &tv1, const CUtensorMap &to, const PrefillParams &p,
                           int d, bool causal, int kind, int grid, cudaStream_t stream,
                           int qtiles) {
  if (kind == kKindVarlen && qtiles == 1)
    return d == 64 ? launch_prefill_k<64, kKindVarlen, 1>(tq, tk, tv, tv1, to, p, causal, grid, stream)
                   : launch_prefill_k<128, kKindVarlen, 1>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  if (d == 64) {
    if (kind == kKindDense)
      return launch_prefill_k<64, kKindDense>(tq, tk, tv, tv1, to, p, causal, grid, stream);
    if (kind == kKindVarlen)
      return launch_prefill_k<64, kKindVarlen>(tq, tk, tv, tv1, to, p, causal, grid, stream);
    if (kind == kKindVarlenHeads)
      return launch_prefill_k<64, kKindVarlenHeads>(tq, tk, tv, tv1, to, p, causal, grid, stream);
    if (kind == kKindDenseHeads)
      return launch_prefill_k<64, kKindDenseHeads>(tq, tk, tv, tv1, to, p, causal, grid, stream);
    if (kind == kKindDenseSplit)
      return launch_prefill_k<64, kKindDenseSplit>(tq, tk, tv, tv1, to, p, causal, grid, stream);
    if (kind == kKindPagedHeads)
      return launch_prefill_k<64, kKindPagedHeads>(tq, tk, tv, tv1, to, p, causal, grid, stream);
    return launch_prefill_k<64, kKindPaged>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  }
  if (kind == kKindDense)
    return launch_prefill_k<128, kKindDense>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  if (kind == kKindVarlen)
    return launch_prefill_k<128, kKindVarlen>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  if (kind == kKindVarlenHeads)
    return launch_prefill_k<128, kKindVarlenHeads>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  if (kind == kKindDenseHeads)
    return launch_prefill_k<128, kKindDenseHeads>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  if (kind == kKindDenseSplit)
    return launch_prefill_k<128, kKindDenseSplit>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  if (kind == kKindPagedHeads)
    return launch_prefill_k<128, kKindPagedHeads>(tq, tk, tv, tv1, to, p, causal, grid, stream);
  return launch_prefill_k<128, kKindPaged>(tq, tk, tv, tv1, to, p, causal, grid, stream);
}

}  // namespace fa
