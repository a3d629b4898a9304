// backward.cu - gradient of exact attention (dQ, dK, dV) for sm_103a.
//
// The pages describe the forward streaming softmax only; the backward pass
// is the chain rule through the same definition, O = softmax(scale Q K^T) V:
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O),
//   dQ = scale dS K,  dK = scale dS^T Q,
// with P recomputed tile by tile from Q, K and the forward log-sum-exp, so
// neither P nor S ever reaches HBM (the same IO argument as the forward).
//
// Three kernels, for dense batches and for packed batches of sequences
// (cu_seqlens; each sequence sees only its own keys):
//   bwd_preprocess   -D and -log-sum-exp in log2 units, per (b, h, row); also
//                    zeroes the work counters of the two kernels after it.
//   bwd_dq           per (b, h, 128-row query tile) work item; streams the
//                    key tiles: S = Q K^T and dP = dO V^T (tcgen05, TMEM),
//                    dS in registers, dQ += dS K (A = dS from TMEM).
//   bwd_dkdv         per (b, kv head, 128-key tile) work item; streams the
//                    query tiles of every query head of the group:
//                    S^T = K Q^T and dP^T = V dO^T, then dV += P^T dO and
//                    dK += dS^T Q (A from TMEM), so the group's sum stays in
//                    TMEM and no atomics are needed.
// bwd_dq and bwd_dkdv are persistent: one CTA per SM claims work items from
// a counter, heaviest first, and every barrier of its pipeline counts tiles
// over all of its items.
// Roles per CTA: warps 0-7 elementwise (warps w and w + 4 share the TMEM
// lanes of rows 32 (w % 4) .. + 31 and take the lower and upper 64 columns),
// warp 8 issues the MMAs (converged, elect.sync), warp 9 claims items and is
// the TMA producer.
// The bf16 operands the elementwise warps write (P, dS) land in the columns
// each half has already read: keys 0-63 in columns [0, 32), keys 64-127 in
// [64, 96) of the region, so the TMEM-sourced MMAs read them at that split.
#include <algorithm>

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "bwd_internal.h"
#include "fa_internal.h"
#include "ptx.cuh"
#include "checks.cuh"

namespace fa {

namespace {

constexpr float kLog2eF = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kChunkBytes = 128 * 128;  // 128 rows x one 128-byte swizzle row
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  // dK/dV kernel: K, V, then a ring of Q tiles (with their log-sum-exp
  // vectors) and a ring of dO tiles (with their D vectors), 128 floats per
  // vector.  Both are released once dK is done (dO's vector is read by the
  // elementwise warps until then); Q gets the deeper ring, because S^T of
  // the next query tile needs it right after dV, a product earlier than
  // dP^T needs dO.
  static constexpr int kStagesQ = 3;
  static constexpr int kStagesO = 2;
  static constexpr int kA = 0;                          // K
  static constexpr int kB = kA + kTileBytes;            // V
  static constexpr int kQ = kB + kTileBytes;            // Q ring
  static constexpr int kDO = kQ + kStagesQ * kTileBytes;  // dO ring
  static constexpr int kVecQ = kDO + kStagesO * kTileBytes;  // -lse2 per Q stage
  static constexpr int kVecO = kVecQ + kStagesQ * 512;       // -D per dO stage
  static constexpr int kBar = kVecO + kStagesO * 512;
  static constexpr int kNumBars = 1 + 2 * kStagesQ + 2 * kStagesO + 9;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kItem = kMisc + 16;  // the work item slot
  static constexpr int kBytes = kItem + 32;
  // Room to align the base up to 1 KiB, as much as the 227 KiB limit leaves
  // at d = 128 (the dynamic shared memory of a kernel without static
  // shared memory starts 1 KiB aligned; the kernel checks).
  static constexpr int kSlack = (kBytes + 1024 <= 232448) ? 1024 : 232448 - kBytes;
  static constexpr int kSmemAlloc = kBytes + kSlack;
  static_assert(kSlack >= 0, "dK/dV shared memory exceeds 227 KiB");
};

// Shared memory of the dQ kernel: Q and dO of the query tile, then separate
// K and V rings (V_j is released as soon as dP_j is done, K_j only after
// dQ_j, so K gets the deeper ring).
template <int D>
struct BwdDqLayout {
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStagesK = 3;
  static constexpr int kStagesV = 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;
  static constexpr int kV = kK + kStagesK * kTileBytes;
  static constexpr int kBar = kV + kStagesV * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 9;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kItem = kMisc + 16;  // the work item slot
  static constexpr int kVec = kItem + 32;   // the item's -lse2 and -D vectors (128 floats each)
  static constexpr int kBytes = kVec + 1024;
  static constexpr int kSmemAlloc = kBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "dQ shared memory exceeds 227 KiB");
};

// S-like MMA (both operands K-major over d): D[tmem] = A[128 x d] B[128 x d]^T.
// One lane of the converged MMA warp (the same one every time) issues the
// whole product; the K-steps advance the descriptors' address fields.
template <int D>
__device__ __forceinline__ void mma_tile_ss(uint32_t d_t, uint32_t a_base, uint32_t b_base) {
  using L = BwdLayout<D>;
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, false, false);
  if (elect_one()) {
    const uint64_t a0 = sdesc_sw128(a_base, 16, 1024), b0 = sdesc_sw128(b_base, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4);
      mma_ss(d_t, a0 + off, b0 + off, kIdesc, kk > 0 ? 1u : 0u);
    }
  }
  __syncwarp();
}

// O-like MMA: D[tmem, 128 x d] (+)= A[tmem, 128 x 128 bf16, split columns] B[128 x d]
// with B a [rows x d] tile read MN-major (the contraction runs over rows).
template <int D>
__device__ __forceinline__ void mma_tile_ts(uint32_t d_t, uint32_t a_t, uint32_t b_base,
                                            bool acc) {
  using L = BwdLayout<D>;
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, D, false, true);
  if (elect_one()) {
    const uint64_t b0 = sdesc_sw128(b_base, L::kChunkBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < 128 / 16; ++kk)
      mma_ts(d_t, a_t + kk * 8 + (kk >= 4 ? 32 : 0),
             b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), kIdesc, (acc || kk > 0) ? 1u : 0u);
  }
  __syncwarp();
}

// Writes one half (D / 2 columns) of the 128 rows of a tile as bf16 times
// `mul`: lane l holds its row's half, fp32 from TMEM in v (32 columns per
// v[c]).  Row by row (one row per lane) a warp's 16-byte stores would touch
// 32 rows at once; instead the lanes of each group of NCH = D / 16 exchange
// 16-byte chunks (an NCH x NCH transpose by xor butterflies), so that store
// i of lane l writes chunk l % NCH of the group's row i and every store
// instruction covers 32 / NCH whole half-rows.  `row_ptr` is this lane's
// half-row, `row_step` the elements from one row to the next (the rows of a
// tile are consecutive); a row whose lane has `row_ok` false is not written.
template <int D>
__device__ __forceinline__ void store_half_rows_bf16(uint16_t *row_ptr, size_t row_step,
                                                     bool row_ok, const uint32_t (&v)[D / 64][32],
                                                     float mul) {
  constexpr int NCH = D / 16;
  const int lane = threadIdx.x & 31;
  uint32_t x[NCH][4];  // chunk c: columns [8c, 8c + 8) of the half
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int k = 8 * c + 2 * w;
      x[c][w] = pack_bf16x2(__uint_as_float(v[k / 32][k % 32]) * mul,
                            __uint_as_float(v[k / 32][k % 32 + 1]) * mul);
    }
  // after the stages lane (base + t) holds chunk t of row (base + c) in x[c]
#pragma unroll
  for (int sft = NCH / 2; sft > 0; sft >>= 1) {
    const bool hi = (lane & sft) != 0;
#pragma unroll
    for (int c0 = 0; c0 < NCH; ++c0) {
      if (c0 & sft) continue;
      const int c1 = c0 | sft;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi ? x[c0][w] : x[c1][w], sft);
        if (hi)
          x[c0][w] = recv;
        else
          x[c1][w] = recv;
      }
    }
  }
  const unsigned ok_rows = __ballot_sync(0xffffffffu, row_ok);
  const int sub = lane % NCH, base = lane - sub;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    if ((ok_rows >> (base + i)) & 1u) {
      uint16_t *dst = row_ptr + static_cast<ptrdiff_t>(base + i - lane) * static_cast<ptrdiff_t>(row_step) +
                      sub * 8;
      *reinterpret_cast<uint4 *>(dst) = make_uint4(x[i][0], x[i][1], x[i][2], x[i][3]);
    }
  }
}

// First row and length of sequence b: in a packed batch from cu_seqlens
// (a sequence with invalid bounds, or longer than N, is reported and gets
// length 0, so nothing of it is computed or written); in a dense batch the
// rows of batch element b (row coordinates are then per element).
template <bool VARLEN>
__device__ __forceinline__ void bwd_seq(const BwdParams &p, int b, int &start, int &len,
                                        bool report) {
  if constexpr (VARLEN) {
    const int a = checked_load(p.cu_seqlens, b, p.B + 1, p.status);
    const int e = checked_load(p.cu_seqlens, b + 1, p.B + 1, p.status);
    if (a < 0 || e < a || e > p.total_tokens || e - a > p.N) {
      if (report) raise_status(p.status, FA_DEV_BAD_SEQLEN);
      start = 0;
      len = 0;
      return;
    }
    start = a;
    len = e - a;
  } else {
    start = 0;
    len = p.N;
  }
}

// Longest-first order of the 128-row tiles of a packed batch of at most
// kBwdOrderMaxSeqs sequences, so that the heaviest CTAs start first and the
// last wave holds the lightest ones.  Levels L = n_tiles .. 1 in turn:
//  - causal: level L holds, for every sequence of at least L tiles (in
//    sequence order), the tile whose work is L tiles: query tile L - 1 (it
//    sees L key tiles) or key tile n_b - L (L query tiles see it);
//  - non-causal: level L holds every tile of the sequences of exactly L tiles
//    (each tile's work is the sequence's n_b tiles).
// Returns the sequence of work item `item` and sets `tile`, or returns -1 past
// the last item.  Run by whole warps (every lane gets the answer); a sequence
// with invalid bounds has no tiles (the preprocess reports it).
template <bool CAUSAL, bool KEY_TILES>
__device__ __forceinline__ int longest_first_item(const BwdParams &p, int item, int &tile) {
  const int lane = threadIdx.x & 31;
  int nt[kBwdOrderMaxSeqs / 32];  // tiles of sequence lane + 32 k
#pragma unroll
  for (int k = 0; k < kBwdOrderMaxSeqs / 32; ++k) {
    const int b = lane + 32 * k;
    nt[k] = 0;
    if (b < p.B) {
      const int a = checked_load(p.cu_seqlens, b, p.B + 1, p.status);
      const int e = checked_load(p.cu_seqlens, b + 1, p.B + 1, p.status);
      if (a >= 0 && e >= a && e <= p.total_tokens && e - a <= p.N) nt[k] = (e - a + 127) / 128;
    }
  }
  // items at levels >= L (non-increasing in L)
  auto above = [&](int L) {
    int c = 0;
#pragma unroll
    for (int k = 0; k < kBwdOrderMaxSeqs / 32; ++k)
      c += CAUSAL ? max(0, nt[k] - L + 1) : (nt[k] >= L ? nt[k] : 0);
#pragma unroll
    for (int sft = 16; sft > 0; sft >>= 1) c += __shfl_xor_sync(0xffffffffu, c, sft);
    return c;
  };
  if (item >= above(1)) return -1;
  int lo = 1, hi = p.n_tiles;  // the level of `item`: the largest L with above(L) > item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (above(mid) > item)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int L = lo;
  int o = item - (L < p.n_tiles ? above(L + 1) : 0);  // place in the level
  int idx = o;                                          // member of the level
  if (!CAUSAL) {
    idx = o / L;
    tile = o % L;
  }
#pragma unroll
  for (int k = 0; k < kBwdOrderMaxSeqs / 32; ++k) {
    const bool in = CAUSAL ? nt[k] >= L : nt[k] == L;
    const unsigned m = __ballot_sync(0xffffffffu, in);
    const int cnt = __popc(m);
    if (idx < cnt) {
      const bool hit = in && __popc(m & ((1u << lane) - 1u)) == idx;
      const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
      const int n_b = __shfl_sync(0xffffffffu, nt[k], src);
      if (CAUSAL) tile = KEY_TILES ? n_b - L : L - 1;
      return src + 32 * k;
    }
    idx -= cnt;
  }
  return -1;  // not reached: the level holds idx + 1 members
}

// A work item of a persistent backward CTA: one 128-row tile of one
// sequence (batch element) and one head, handed from the producer warp to
// the others through shared memory.
struct BwdItem {
  int b;      // sequence
  int tile;   // query tile (dQ) or key tile (dK / dV)
  int h;      // query head (dQ) or KV head (dK / dV)
  int start;  // the sequence's first row in a packed batch (0 when dense)
  int len;    // its rows
  int valid;  // 0: no work left
};
static_assert(sizeof(BwdItem) <= 32, "work item slot");

// Claims the next work item from the call's counter (lane 0 takes an index,
// the whole warp decodes it) and returns it, or an item with valid = 0 once
// none are left.  Heads run fastest.  Tiles run heaviest first: for the
// query tiles of a causal pass the last tile first, for key tiles the first;
// a dense batch takes sequence by sequence, a packed batch its tiles
// longest-first; a packed batch of more sequences than that order covers
// takes sequence by sequence and claims again past a sequence's last tile.
// Run by whole warps.
template <bool CAUSAL, bool VARLEN, bool KEY_TILES>
__device__ BwdItem claim_item(const BwdParams &p, unsigned int *counter, int heads) {
  BwdItem it{};
  const long long total = static_cast<long long>(p.B) * p.n_tiles * heads;
  for (;;) {
    unsigned int w = 0;
    if ((threadIdx.x & 31) == 0) w = atomicAdd(counter, 1u);
    w = __shfl_sync(0xffffffffu, w, 0);
    if (w >= total) return it;
    const int h = static_cast<int>(w % heads);
    const int r = static_cast<int>(w / heads);
    int b, rank, t;
    if (VARLEN && p.longest_first) {
      b = longest_first_item<CAUSAL, KEY_TILES>(p, r, t);
      if (b < 0) return it;
    } else {
      // sequence by sequence (the items in flight share the sequence's K and
      // V, or Q and dO, in L2)
      b = r / p.n_tiles;
      rank = r % p.n_tiles;
      t = (CAUSAL && !KEY_TILES) ? p.n_tiles - 1 - rank : rank;
    }
    int start, len;
    bwd_seq<VARLEN>(p, b, start, len, false);
    if (t < (len + 127) / 128) {
      it.b = b;
      it.tile = t;
      it.h = h;
      it.start = start;
      it.len = len;
      it.valid = 1;
      return it;
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ preprocess
// D / 8 threads per (b, row, h), 16 bytes each: D = sum_c dO * O (fp32 from
// bf16) and the forward log-sum-exp in log2 units, both stored negated (the
// consumers add them); -lse is -inf for rows past N or rows without a visible
// key, so that every weight recomputed from it is 0.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  constexpr int TPR = D / 8;  // threads per row
  const int sub = threadIdx.x % TPR;
  const long long gr = static_cast<long long>(blockIdx.x) * (256 / TPR) + threadIdx.x / TPR;
  const long long total = static_cast<long long>(p.B) * p.Npad * p.H;
  // the work counters of the dQ and dK / dV kernels, which run after this one
  if (blockIdx.x == 0 && threadIdx.x < 2) p.work[threadIdx.x] = 0u;
  if (gr >= total) return;  // whole row groups leave together (TPR divides 32)
  // Row groups run over the rows of one (b, h) first, so that the lse reads
  // and the D / lse2 writes of a warp are contiguous; each row's O and dO
  // are still read as whole 16-byte chunks.
  const int row = static_cast<int>(gr % p.Npad);
  const long long bh = gr / p.Npad;
  const int h = static_cast<int>(bh % p.H);
  const int b = static_cast<int>(bh / p.H);
  const size_t vec = static_cast<size_t>(gr);  // (b * H + h) * Npad + row
  // elements of O / dO, and of the workspace vectors, the call owns
  const size_t n_rows =
      VARLEN ? static_cast<size_t>(p.total_tokens) * p.H : static_cast<size_t>(p.B) * p.N * p.H;
  const size_t n_vec = static_cast<size_t>(p.B) * p.H * p.Npad;
  int start, len;
  bwd_seq<VARLEN>(p, b, start, len, row == 0 && h == 0 && sub == 0);
  // the row's place in O / dO and in the log-sum-exp
  const size_t grow = VARLEN ? static_cast<size_t>(start) + row : static_cast<size_t>(b) * p.N + row;
  const size_t lidx = VARLEN ? static_cast<size_t>(h) * p.total_tokens + start + row
                             : (static_cast<size_t>(b) * p.H + h) * p.N + row;
  float acc = 0.f;
  const size_t off = (grow * p.H + h) * D + sub * 8;
  if (row < len && in_bounds(off, 8, n_rows * D, p.status)) {
    const uint4 o = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.out) + off);
    const uint4 g = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.dout) + off);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a2 = bf16x2_to_float2(ow[e]);
      const float2 c2 = bf16x2_to_float2(gw[e]);
      acc = fmaf(a2.x, c2.x, acc);
      acc = fmaf(a2.y, c2.y, acc);
    }
  }
#pragma unroll
  for (int sft = TPR / 2; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
  if (sub == 0 && in_bounds(vec, 1, n_vec, p.status)) {
    if (row < len) {
      const float l = checked_load(p.lse, lidx, n_rows, p.status);
      p.nlse2[vec] = (l == -CUDART_INF_F) ? -CUDART_INF_F : -(l * kLog2eF);
      p.ndsum[vec] = -acc;
    } else {
      p.nlse2[vec] = -CUDART_INF_F;
      p.ndsum[vec] = 0.f;
    }
  }
}

// ------------------------------------------------------------------------- dQ
// Persistent: one CTA per SM takes (query tile, head) work items from the
// call's counter until none are left, so that one item's first products and
// copies overlap the previous item's dQ epilogue and no CTA launch or set-up
// sits between items.  The producer warp claims and decodes each item and
// hands it to the other warps through shared memory (slot, published by the
// Q / dO barrier); every barrier of the key-tile pipeline counts key tiles
// over all of the CTA's items.
template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdParams p) {
  using L = BwdDqLayout<D>;
  constexpr int SK = L::kStagesK;
  constexpr int SV = L::kStagesV;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint64_t *in_full = bars;        // Q and dO of the item (and its slot)
  uint64_t *k_full = bars + 1;     // [SK]
  uint64_t *k_empty = k_full + SK;
  uint64_t *v_full = k_empty + SK;  // [SV]
  uint64_t *v_empty = v_full + SV;
  uint64_t *s_full = v_empty + SV;
  uint64_t *s_read = s_full + 1;    // the elementwise warps have read S_j
  uint64_t *dp_full = s_read + 1;
  uint64_t *p_full = dp_full + 1;   // dS_j (bf16) is in TMEM
  uint64_t *dq_done = p_full + 1;   // the item's dQ is complete in TMEM
  uint64_t *drain = dq_done + 1;
  uint64_t *qdo_empty = drain + 1;  // the item's last products that read Q and dO are done
  uint64_t *dq_free = qdo_empty + 1;  // the elementwise warps have read the item's dQ
  uint64_t *taken = dq_free + 1;    // the MMA and elementwise warps have read the slot
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
  volatile BwdItem *slot = reinterpret_cast<volatile BwdItem *>(smem + L::kItem);
  float *sVec = reinterpret_cast<float *>(smem + L::kVec);  // -lse2 [0, 128), -D [128, 256)
  uint8_t *sQ = smem + L::kQ;
  uint8_t *sDO = smem + L::kDO;
  uint8_t *sK = smem + L::kK;
  uint8_t *sV = smem + L::kV;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (warp == 9 && lane == 0) {
    mbar_init(in_full, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, 256);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 256);
    mbar_init(dq_done, 1);
    mbar_init(drain, 1);
    mbar_init(qdo_empty, 1);
    mbar_init(dq_free, 256);
    mbar_init(taken, 9);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // reads the slot of item m (and, for row `row` >= 0, its entries of the
  // item's vectors) once its barrier phase is complete, then tells the
  // producer (one arrival per warp)
  auto take = [&](int m, BwdItem &it, int row, float &nlse2, float &ndsum) -> bool {
    bool ok = mbar_wait(in_full, m & 1, abort_flag, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    it.b = slot->b;
    it.tile = slot->tile;
    it.h = slot->h;
    it.start = slot->start;
    it.len = slot->len;
    it.valid = slot->valid;
    if (row >= 0 && it.valid) {
      nlse2 = sVec[row];
      ndsum = sVec[128 + row];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(taken);
    return true;
  };

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    // Item m: claim and decode it, wait until every warp has read slot m - 1
    // and the products of item m - 1 that read Q and dO are done, publish
    // it with its Q and dO, then K(j) and V(j) of its key tiles, each ring
    // counting key tiles over all items.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    bool ok = true;
    int gk = 0, gv = 0;  // K and V tiles issued so far
    int last = -1;       // the last item whose Q and dO were issued
    for (int m = 0;; ++m) {
      const BwdItem it = claim_item<CAUSAL, VARLEN, false>(p, p.work + 0, p.H);
      if (lane == 0 && m > 0)
        ok = mbar_wait(taken, (m - 1) & 1, abort_flag, p.status) &&
             mbar_wait(qdo_empty, (m - 1) & 1, abort_flag, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        slot->b = it.b;
        slot->tile = it.tile;
        slot->h = it.h;
        slot->start = it.start;
        slot->len = it.len;
        slot->valid = it.valid;
        if (it.valid) {
          const int row0 = VARLEN ? it.start : 0, bc = VARLEN ? 0 : it.b;
          // the tile's 128 entries of the workspace vectors (a checked build
          // that finds them outside the workspace copies entries 0..127, so
          // that the barrier still gets its bytes)
          size_t vec = (static_cast<size_t>(it.b) * p.H + it.h) * p.Npad + it.tile * 128;
          if (!in_bounds(vec, 128, static_cast<size_t>(p.B) * p.H * p.Npad, p.status)) vec = 0;
          mbar_arrive_expect_tx(in_full, 2 * L::kTileBytes + 1024);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_4d(sQ + c * L::kChunkBytes, &tm_q, in_full, c * 64, it.h, row0 + it.tile * 128, bc);
            tma_load_4d(sDO + c * L::kChunkBytes, &tm_do, in_full, c * 64, it.h, row0 + it.tile * 128,
                        bc);
          }
          bulk_load(sVec, p.nlse2 + vec, 512, in_full);
          bulk_load(sVec + 128, p.ndsum + vec, 512, in_full);
        } else {
          mbar_arrive(in_full);  // no work left: publishes the empty slot
        }
      }
      if (!it.valid) break;
      last = m;
      if (lane == 0) {
        const int row0 = VARLEN ? it.start : 0, bc = VARLEN ? 0 : it.b;
        const int kvh = it.h / p.group;
        const int n_kv = CAUSAL ? it.tile + 1 : (it.len + 127) / 128;
        for (int j = 0; j < n_kv; ++j) {
          const int sk = gk % SK, sv = gv % SV;
          if (gk >= SK && !mbar_wait(&k_empty[sk], ((gk / SK) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[sk], L::kTileBytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(sK + sk * L::kTileBytes + c * L::kChunkBytes, &tm_k, &k_full[sk], c * 64,
                        kvh, row0 + j * 128, bc);
          ++gk;
          if (gv >= SV && !mbar_wait(&v_empty[sv], ((gv / SV) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[sv], L::kTileBytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(sV + sv * L::kTileBytes + c * L::kChunkBytes, &tm_v, &v_full[sv], c * 64,
                        kvh, row0 + j * 128, bc);
          ++gv;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
    }
    if (!ok && lane == 0) {
      // a wait ran out: let the copies still in flight land before the CTA
      // leaves (Q and dO of the last item, K and V of the last tiles issued)
      if (last >= 0) mbar_drain(in_full, last & 1, p.status);
      for (int x = max(0, gk - SK); x < gk; ++x) mbar_drain(&k_full[x % SK], (x / SK) & 1, p.status);
      for (int x = max(0, gv - SV); x < gv; ++x) mbar_drain(&v_full[x % SV], (x / SV) & 1, p.status);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // S lives in TMEM [0,128), dQ in [256, 256 + d), and dP in two buffers,
    // [128,256) for even key tiles and [384,512) for odd ones (key tiles
    // counted over the CTA's items).  Per key tile j: S_{j+1} as soon as the
    // elementwise warps have read S_j (s_read), then dP_{j+1} into the other
    // buffer, so both run while they finish tile j; then dQ += dS_j K_j once
    // dS_j (bf16, written over dP_j) is in TMEM.  dP_{j+2} takes dS_j's
    // buffer only after dQ_j, issued before it by this thread, has read it.
    // An item's S_0 and dP_0 are issued while the elementwise warps still
    // store the previous item's dQ; its first dQ product waits for them to
    // have read it (dq_free).
    const uint32_t q_base = smem_u32(sQ), do_base = smem_u32(sDO);
    const uint32_t k_ring = smem_u32(sK), v_ring = smem_u32(sV);
    auto issue_s = [&](int g) -> bool {
      const int sk = g % SK;
      if (!mbar_wait_warp(&k_full[sk], (g / SK) & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      mma_tile_ss<D>(tmem, q_base, k_ring + sk * L::kTileBytes);
      mma_commit_elect(s_full);
      return true;
    };
    auto issue_dp = [&](int g) -> bool {
      const int sv = g % SV;
      if (!mbar_wait_warp(&v_full[sv], (g / SV) & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      mma_tile_ss<D>(tmem + ((g & 1) ? 384 : 128), do_base, v_ring + sv * L::kTileBytes);
      mma_commit_elect(dp_full);
      mma_commit_elect(&v_empty[sv]);
      return true;
    };
    bool ok = true;
    int g0 = 0;  // key tiles of the earlier items
    for (int m = 0; ok; ++m) {
      BwdItem it;
      float unused0, unused1;
      if (!take(m, it, -1, unused0, unused1) || !it.valid) break;
      const int n_kv = CAUSAL ? it.tile + 1 : (it.len + 127) / 128;
      tc_fence_after();
      ok = issue_s(g0) && issue_dp(g0);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int g = g0 + j;
        if (j + 1 < n_kv) {
          ok = mbar_wait_warp(s_read, g & 1, abort_flag, p.status) && issue_s(g + 1) &&
               issue_dp(g + 1);
          if (!ok) break;
        } else {
          mma_commit_elect(qdo_empty);  // the item's last S and dP read Q and dO
        }
        if (!mbar_wait_warp(p_full, g & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (j == 0 && m > 0 && !mbar_wait_warp(dq_free, (m - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_tile_ts<D>(tmem + 256, tmem + ((g & 1) ? 384 : 128), k_ring + (g % SK) * L::kTileBytes,
                       j > 0);
        mma_commit_elect(&k_empty[g % SK]);
      }
      if (!ok) break;
      mma_commit_elect(dq_done);
      g0 += n_kv;
    }
    mma_commit_elect(drain);
    mbar_drain(drain, 0, p.status);
  } else {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3, hf = warp >> 2;  // TMEM lane group, column half
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off, tQ = tmem + 256 + lane_off;
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    bool ok = true;
    int g0 = 0;
    for (int m = 0; ok; ++m) {
      BwdItem it;
      float nlse2 = 0.f, ndsum = 0.f;  // -lse (log2 units) and -D of the row
      if (!take(m, it, row, nlse2, ndsum) || !it.valid) break;
      const int qi = it.tile * 128 + row;
      const int len = it.len;
      const int n_kv = CAUSAL ? it.tile + 1 : (len + 127) / 128;
      const float2 nl2 = make_float2(nlse2, nlse2), nd2 = make_float2(ndsum, ndsum);
      for (int j = 0; j < n_kv; ++j) {
        const int g = g0 + j;
        ok = mbar_wait(s_full, g & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // keys [0, nvis) of this tile are visible to the row (keys past the
        // sequence, of the next sequence in a packed batch, are not)
        const int nvis = min(128, (CAUSAL ? min(len, qi + 1) : len) - j * 128);
        // P = exp(S * scale - lse) of this half's 64 keys, kept as bf16 pairs
        // (the values the dQ product uses through dS)
        // (packed pairs; the mask is applied only in chunks that reach past nvis)
        uint32_t pp[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          uint32_t sv[32];
          tmem_ld32_wait(tS + c * 32, sv);
          const bool part = c * 32 + 32 > nvis;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 x =
                ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2x2, nl2);
            float w0 = ex2(x.x), w1 = ex2(x.y);
            if (part) {
              w0 = (c * 32 + e < nvis) ? w0 : 0.f;
              w1 = (c * 32 + e + 1 < nvis) ? w1 : 0.f;
            }
            pp[cc * 16 + (e >> 1)] = pack_bf16x2(w0, w1);
          }
        }
        tc_fence_before();
        mbar_arrive(s_read);
        ok = mbar_wait(dp_full, g & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // dS = P (dP - D), written over this half's dP columns (dP_j in the
        // buffer of key tile j's parity)
        const uint32_t tP = tmem + ((g & 1) ? 384 : 128) + lane_off;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          uint32_t dp[32], pk[16];
          tmem_ld32_wait(tP + c * 32, dp);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 w = bf16x2_to_float2(pp[cc * 16 + (e >> 1)]);
            const float2 r = fmul2(
                w, fadd2(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2));
            pk[e >> 1] = pack_bf16x2(r.x, r.y);
          }
          tmem_st16(tP + hf * 64 + cc * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      ok = mbar_wait(dq_done, m & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // this half's dQ columns into registers, TMEM handed back, then the row
      uint32_t o[D / 64][32];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tmem_ld32_wait(tQ + (hf * (D / 64) + c) * 32, o[c]);
      tc_fence_before();
      mbar_arrive(dq_free);
      const size_t grow =
          VARLEN ? static_cast<size_t>(it.start) + qi : static_cast<size_t>(it.b) * p.N + qi;
      const size_t drow = (grow * p.H + it.h) * D;
      const size_t rows = VARLEN ? static_cast<size_t>(p.total_tokens) : static_cast<size_t>(p.B) * p.N;
      const bool row_ok = qi < len && in_bounds(drow, D, rows * p.H * D, p.status);
      store_half_rows_bf16<D>(static_cast<uint16_t *>(p.dq) + drow + hf * (D / 2),
                              static_cast<size_t>(p.H) * D, row_ok, o, p.scale);
      g0 += n_kv;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------- dK dV
// Persistent like the dQ kernel: one CTA per SM takes (key tile, KV head)
// items from the call's second counter.  An item's K and V stay resident;
// the Q and dO rings (with their vectors) and every barrier of the
// iteration pipeline count iterations over all of the CTA's items, so the
// next item's copies and its first S^T and dP^T overlap the previous item's
// last products and its dV / dK epilogue.
template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using L = BwdLayout<D>;
  constexpr int SQ = L::kStagesQ;
  constexpr int SO = L::kStagesO;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (smem - smem_raw > L::kSlack) {
    // the layout does not fit: report it, touch nothing (the whole CTA leaves)
    if (threadIdx.x == 0) raise_status(p.status, FA_DEV_SMEM_ALIGN);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint64_t *in_full = bars;          // K and V of the item (and its slot)
  uint64_t *q_full = bars + 1;       // [SQ] Q and its -lse2 vector
  uint64_t *q_empty = q_full + SQ;
  uint64_t *o_full = q_empty + SQ;   // [SO] dO and its -D vector
  uint64_t *o_empty = o_full + SO;
  uint64_t *s_full = o_empty + SO;
  uint64_t *dp_full = s_full + 1;
  uint64_t *pt_full = dp_full + 1;  // P^T (bf16) is in TMEM
  uint64_t *p_full = pt_full + 1;   // dS^T (bf16) is in TMEM
  uint64_t *kv_done = p_full + 1;   // the item's dV and dK are complete in TMEM
  uint64_t *drain = kv_done + 1;
  uint64_t *kv_empty = drain + 1;   // the item's last products that read K and V are done
  uint64_t *kv_free = kv_empty + 1;  // the elementwise warps have read the item's dV and dK
  uint64_t *taken = kv_free + 1;    // the MMA and elementwise warps have read the slot
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
  volatile BwdItem *slot = reinterpret_cast<volatile BwdItem *>(smem + L::kItem);
  uint8_t *sK = smem + L::kA;
  uint8_t *sV = smem + L::kB;
  uint8_t *sQr = smem + L::kQ;    // Q ring
  uint8_t *sOr = smem + L::kDO;   // dO ring
  float *sVq = reinterpret_cast<float *>(smem + L::kVecQ);  // Q stage s: -lse2 at 128 s
  float *sVo = reinterpret_cast<float *>(smem + L::kVecO);  // dO stage s: -D at 128 s

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (warp == 9 && lane == 0) {
    mbar_init(in_full, 1);
    for (int s = 0; s < SQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < SO; ++s) {
      mbar_init(&o_full[s], 1);
      mbar_init(&o_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(pt_full, 256);
    mbar_init(p_full, 256);
    mbar_init(kv_done, 1);
    mbar_init(drain, 1);
    mbar_init(kv_empty, 1);
    mbar_init(kv_free, 256);
    mbar_init(taken, 9);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // reads the slot of item m once its barrier phase is complete, then tells
  // the producer (one arrival per warp)
  auto take = [&](int m, BwdItem &it) -> bool {
    bool ok = mbar_wait(in_full, m & 1, abort_flag, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    it.b = slot->b;
    it.tile = slot->tile;
    it.h = slot->h;
    it.start = slot->start;
    it.len = slot->len;
    it.valid = slot->valid;
    __syncwarp();
    if (lane == 0) mbar_arrive(taken);
    return true;
  };
  // iterations of an item: its query tiles that see a key of the tile
  // (from the key tile on, causal) times the query heads of the KV head;
  // iteration it is query head kvh * group + it % group, query tile
  // i0 + it / group
  auto iterations = [&](const BwdItem &it) {
    return ((it.len + 127) / 128 - (CAUSAL ? it.tile : 0)) * p.group;
  };

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    bool ok = true;
    int gq = 0, go = 0;  // Q and dO stages issued so far
    int last = -1;       // the last item whose K and V were issued
    for (int m = 0;; ++m) {
      const BwdItem it = claim_item<CAUSAL, VARLEN, true>(p, p.work + 1, p.Hkv);
      if (lane == 0 && m > 0)
        ok = mbar_wait(taken, (m - 1) & 1, abort_flag, p.status) &&
             mbar_wait(kv_empty, (m - 1) & 1, abort_flag, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        slot->b = it.b;
        slot->tile = it.tile;
        slot->h = it.h;
        slot->start = it.start;
        slot->len = it.len;
        slot->valid = it.valid;
        if (it.valid) {
          const int row0 = VARLEN ? it.start : 0, bc = VARLEN ? 0 : it.b;
          mbar_arrive_expect_tx(in_full, 2 * L::kTileBytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_4d(sK + c * L::kChunkBytes, &tm_k, in_full, c * 64, it.h, row0 + it.tile * 128, bc);
            tma_load_4d(sV + c * L::kChunkBytes, &tm_v, in_full, c * 64, it.h, row0 + it.tile * 128, bc);
          }
        } else {
          mbar_arrive(in_full);  // no work left: publishes the empty slot
        }
      }
      if (!it.valid) break;
      last = m;
      if (lane == 0) {
        const int row0 = VARLEN ? it.start : 0, bc = VARLEN ? 0 : it.b;
        const int i0 = CAUSAL ? it.tile : 0;
        const int n_it = iterations(it);
        for (int x = 0; x < n_it; ++x) {
          const int hq = it.h * p.group + x % p.group;
          const int i = i0 + x / p.group;
          // (a checked build that finds the 128 entries outside the workspace
          // copies entries 0..127 instead, so the barrier still gets its bytes)
          size_t vec = (static_cast<size_t>(it.b) * p.H + hq) * p.Npad + i * 128;
          if (!in_bounds(vec, 128, static_cast<size_t>(p.B) * p.H * p.Npad, p.status)) vec = 0;
          const int sq = gq % SQ, so = go % SO;
          if (gq >= SQ && !mbar_wait(&q_empty[sq], ((gq / SQ) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[sq], L::kTileBytes + 512);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(sQr + sq * L::kTileBytes + c * L::kChunkBytes, &tm_q, &q_full[sq], c * 64, hq,
                        row0 + i * 128, bc);
          bulk_load(sVq + 128 * sq, p.nlse2 + vec, 512, &q_full[sq]);
          ++gq;
          if (go >= SO && !mbar_wait(&o_empty[so], ((go / SO) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&o_full[so], L::kTileBytes + 512);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(sOr + so * L::kTileBytes + c * L::kChunkBytes, &tm_do, &o_full[so], c * 64,
                        hq, row0 + i * 128, bc);
          bulk_load(sVo + 128 * so, p.ndsum + vec, 512, &o_full[so]);
          ++go;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
    }
    if (!ok && lane == 0) {
      // a wait ran out: let the copies still in flight land before the CTA
      // leaves (K and V of the last item, Q and dO of the last stages issued)
      if (last >= 0) mbar_drain(in_full, last & 1, p.status);
      for (int x = max(0, gq - SQ); x < gq; ++x) mbar_drain(&q_full[x % SQ], (x / SQ) & 1, p.status);
      for (int x = max(0, go - SO); x < go; ++x) mbar_drain(&o_full[x % SO], (x / SO) & 1, p.status);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // S^T lives in TMEM [0,128), dP^T in [128,256), dV and dK after them.
    // Per iteration: dV += P^T dO once P^T (bf16, over S^T) is in TMEM; then
    // S^T of the next iteration (issued after dV by this thread, so it
    // overwrites P^T only after dV has read it); dK += dS^T Q once dS^T
    // (over dP^T) is in TMEM; then dP^T of the next iteration.  An item's
    // first S^T and dP^T are issued while the elementwise warps still store
    // the previous item's dV and dK; its first dV product waits for them to
    // have read both (kv_free).
    const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV);
    auto q_at = [&](int g) { return smem_u32(sQr + (g % SQ) * L::kTileBytes); };
    auto do_at = [&](int g) { return smem_u32(sOr + (g % SO) * L::kTileBytes); };
    bool ok = true;
    int g0 = 0;  // iterations of the earlier items
    for (int m = 0; ok; ++m) {
      BwdItem it;
      if (!take(m, it) || !it.valid) break;
      const int n_it = iterations(it);
      ok = mbar_wait_warp(&q_full[g0 % SQ], (g0 / SQ) & 1, abort_flag, p.status) &&
           mbar_wait_warp(&o_full[g0 % SO], (g0 / SO) & 1, abort_flag, p.status);
      if (!ok) break;
      tc_fence_after();
      mma_tile_ss<D>(tmem, k_base, q_at(g0));
      mma_commit_elect(s_full);
      mma_tile_ss<D>(tmem + 128, v_base, do_at(g0));
      mma_commit_elect(dp_full);
      if (n_it == 1) mma_commit_elect(kv_empty);  // the item's last S^T and dP^T read K and V
      for (int x = 0; x < n_it; ++x) {
        const int g = g0 + x;
        if (!mbar_wait_warp(pt_full, g & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (x == 0 && m > 0 && !mbar_wait_warp(kv_free, (m - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_tile_ts<D>(tmem + 256, tmem, do_at(g), x > 0);
        if (x + 1 < n_it) {
          if (!mbar_wait_warp(&q_full[(g + 1) % SQ], ((g + 1) / SQ) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_ss<D>(tmem, k_base, q_at(g + 1));
          mma_commit_elect(s_full);
        }
        if (!mbar_wait_warp(p_full, g & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_tile_ts<D>(tmem + 256 + D, tmem + 128, q_at(g), x > 0);
        // Q(g) was last read by dK(g); the dO stage is released here too,
        // because the elementwise warps read its -D vector until dS^T(g) is
        // handed over (which dK(g) waited for)
        mma_commit_elect(&q_empty[g % SQ]);
        mma_commit_elect(&o_empty[g % SO]);
        if (x + 1 < n_it) {
          if (!mbar_wait_warp(&o_full[(g + 1) % SO], ((g + 1) / SO) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_ss<D>(tmem + 128, v_base, do_at(g + 1));
          mma_commit_elect(dp_full);
          if (x + 2 == n_it) mma_commit_elect(kv_empty);
        }
      }
      if (!ok) break;
      mma_commit_elect(kv_done);
      g0 += n_it;
    }
    mma_commit_elect(drain);
    mbar_drain(drain, 0, p.status);
  } else {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3, hf = warp >> 2;  // TMEM lane group, column half
    const int row = quad * 32 + lane;   // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off, tP = tmem + 128 + lane_off;
    const uint32_t tV = tmem + 256 + lane_off, tK = tmem + 256 + D + lane_off;
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    bool ok = true;
    int g0 = 0;
    for (int m = 0; ok; ++m) {
      BwdItem itm;
      if (!take(m, itm) || !itm.valid) break;
      const int kj = itm.tile * 128 + row;
      const int len = itm.len;
      const int i0 = CAUSAL ? itm.tile : 0;
      const int n_it = iterations(itm);
      for (int x = 0; x < n_it; ++x) {
        const int g = g0 + x;
        const int i = i0 + x / p.group;
        // the stages' vectors arrived with their tiles (async copies): observe
        // those barriers too before reading them
        ok = mbar_wait(&q_full[g % SQ], (g / SQ) & 1, abort_flag, p.status) &&
             mbar_wait(s_full, g & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float *vl = sVq + 128 * (g % SQ);  // -log-sum-exp (log2 units) of the 128 queries
        const float *vd = sVo + 128 * (g % SO);  // -D of the 128 queries (read after o_full)
        // queries [qfirst, 128) of this tile see the key (causal); earlier
        // ones do not.  Queries past the sequence carry -lse2 = -inf, so
        // their weight is 0.
        const int qfirst = CAUSAL ? max(0, kj - i * 128) : 0;
        // P^T = exp(S^T * scale - lse[q]) of this half's 64 queries as bf16
        // pairs, stored over S^T (packed pairs; the mask is applied only in
        // chunks that start before qfirst)
        uint32_t pp[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          uint32_t sv[32];
          tmem_ld32_wait(tS + c * 32, sv);
          const bool part = c * 32 < qfirst;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int q0 = c * 32 + e;
            const float4 l4 = *reinterpret_cast<const float4 *>(vl + q0);
            const float2 x0 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                    sl2x2, make_float2(l4.x, l4.y));
            const float2 x1 = ffma2(make_float2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])),
                                    sl2x2, make_float2(l4.z, l4.w));
            float w0 = ex2(x0.x), w1 = ex2(x0.y), w2 = ex2(x1.x), w3 = ex2(x1.y);
            if (part) {
              w0 = (q0 >= qfirst) ? w0 : 0.f;
              w1 = (q0 + 1 >= qfirst) ? w1 : 0.f;
              w2 = (q0 + 2 >= qfirst) ? w2 : 0.f;
              w3 = (q0 + 3 >= qfirst) ? w3 : 0.f;
            }
            pp[cc * 16 + (e >> 1)] = pack_bf16x2(w0, w1);
            pp[cc * 16 + (e >> 1) + 1] = pack_bf16x2(w2, w3);
          }
          uint32_t chunk[16];
#pragma unroll
          for (int t2 = 0; t2 < 16; ++t2) chunk[t2] = pp[cc * 16 + t2];
          tmem_st16(tS + hf * 64 + cc * 16, chunk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(pt_full);
        ok = mbar_wait(&o_full[g % SO], (g / SO) & 1, abort_flag, p.status) &&
             mbar_wait(dp_full, g & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // dS^T = P^T (dP^T - D[q]), stored over this half's dP^T columns
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          uint32_t dp[32], pd[16];
          tmem_ld32_wait(tP + c * 32, dp);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int q0 = c * 32 + e;
            const float4 d4 = *reinterpret_cast<const float4 *>(vd + q0);
            const float2 wa = bf16x2_to_float2(pp[cc * 16 + (e >> 1)]);
            const float2 wb = bf16x2_to_float2(pp[cc * 16 + (e >> 1) + 1]);
            const float2 ra = fmul2(
                wa, fadd2(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                          make_float2(d4.x, d4.y)));
            const float2 rb = fmul2(
                wb, fadd2(make_float2(__uint_as_float(dp[e + 2]), __uint_as_float(dp[e + 3])),
                          make_float2(d4.z, d4.w)));
            pd[e >> 1] = pack_bf16x2(ra.x, ra.y);
            pd[(e >> 1) + 1] = pack_bf16x2(rb.x, rb.y);
          }
          tmem_st16(tP + hf * 64 + cc * 16, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      ok = mbar_wait(kv_done, m & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // key rows past the sequence (the next sequence's, in a packed batch)
      // are not written; dV, then dK (TMEM handed back once both are read)
      const size_t grow =
          VARLEN ? static_cast<size_t>(itm.start) + kj : static_cast<size_t>(itm.b) * p.N + kj;
      const size_t orow = (grow * p.Hkv + itm.h) * D;
      const size_t rows = VARLEN ? static_cast<size_t>(p.total_tokens) : static_cast<size_t>(p.B) * p.N;
      const bool row_ok = kj < len && in_bounds(orow, D, rows * p.Hkv * D, p.status);
      const size_t step = static_cast<size_t>(p.Hkv) * D;
      uint32_t o[D / 64][32];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tmem_ld32_wait(tV + (hf * (D / 64) + c) * 32, o[c]);
      store_half_rows_bf16<D>(static_cast<uint16_t *>(p.dv) + orow + hf * (D / 2), step, row_ok, o,
                              1.f);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tmem_ld32_wait(tK + (hf * (D / 64) + c) * 32, o[c]);
      tc_fence_before();
      mbar_arrive(kv_free);
      store_half_rows_bf16<D>(static_cast<uint16_t *>(p.dk) + orow + hf * (D / 2), step, row_ok, o,
                              p.scale);
      g0 += n_it;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------- launch

template <int D, bool VARLEN>
static cudaError_t launch_bwd_d(const CUtensorMap &tq, const CUtensorMap &tdo,
                                const CUtensorMap &tk, const CUtensorMap &tv, const BwdParams &p,
                                bool causal, cudaStream_t stream) {
  using L = BwdLayout<D>;
  const long long pre_rows = static_cast<long long>(p.B) * p.Npad * p.H;
  const long long rows_per_block = 256 / (D / 8);
  bwd_preprocess_kernel<D, VARLEN>
      <<<static_cast<unsigned>((pre_rows + rows_per_block - 1) / rows_per_block), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto dq = causal ? bwd_dq_kernel<D, true, VARLEN> : bwd_dq_kernel<D, false, VARLEN>;
  auto dkdv = causal ? bwd_dkdv_kernel<D, true, VARLEN> : bwd_dkdv_kernel<D, false, VARLEN>;
  e = cudaFuncSetAttribute(dq, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdDqLayout<D>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  // work items: every (sequence, 128-row tile); the longest-first order of a
  // packed batch enumerates only real tiles, at most ceil(T / 128) + B
  long long items = static_cast<long long>(p.B) * p.n_tiles;
  if (VARLEN && p.longest_first)
    items = std::min(items, (p.total_tokens + 127LL) / 128 + p.B);
  const unsigned grid_kv = static_cast<unsigned>(std::min<long long>(items * p.Hkv, p.num_ctas));
  dkdv<<<grid_kv, kBwdThreads, L::kSmemAlloc, stream>>>(tq, tdo, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM at most
  const unsigned grid_q = static_cast<unsigned>(std::min<long long>(items * p.H, p.num_ctas));
  dq<<<grid_q, kBwdThreads, BwdDqLayout<D>::kSmemAlloc, stream>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                       const CUtensorMap &tv, const BwdParams &p, int d, bool causal,
                       cudaStream_t stream) {
  if (p.cu_seqlens != nullptr)
    return d == 64 ? launch_bwd_d<64, true>(tq, tdo, tk, tv, p, causal, stream)
                   : launch_bwd_d<128, true>(tq, tdo, tk, tv, p, causal, stream);
  return d == 64 ? launch_bwd_d<64, false>(tq, tdo, tk, tv, p, causal, stream)
                 : launch_bwd_d<128, false>(tq, tdo, tk, tv, p, causal, stream);
}

}  // namespace fa
