// decode.cu - paged GQA flash-decoding for sm_103a.
//
// "S12 FlashAttention", section "How this composes with what you already
// built": one loop that walks the block table, loads the KV head shared by a
// group of query heads, scores the block and updates (m, l, o).  Section
// "What this unlocks beyond speed" (flash-decoding): with one query token
// there is no parallelism over queries, so the keys of a sequence are split
// across thread blocks, each producing a partial (m, l, o), and a second
// kernel merges the partial states with the same rescaling as the tile
// recurrence (explainer page, "Show the maths").
//
// decode_split_kernel: one warp per (sequence, KV head, split of the
// context).  The 16-token KV blocks named by the block table are fetched
// with TMA (128-byte swizzle) into a ring of shared-memory stages, several
// blocks in flight per warp.  Per block:
//   S^T [16 tokens x 8 heads] = K_blk [16 x d] . Q^T   (mma.m16n8k16, the G
//       query heads of the group are the N columns, padded to 8)
//   column-wise online softmax over the 16 tokens (warp shuffles)
//   O^T [d x 8] += V_blk^T [d x 16] . P^T [16 x 8]     (P^T re-laid out with
//       movmatrix from the S^T accumulator layout)
// The work is bound by HBM reads of K and V; the tensor-core ops are a small
// fraction of the issue slots.
//
// decode_combine_kernel: one CTA per (sequence, query head) merges the
// partial states: M = max m_i, L = sum 2^(m_i - M) l_i,
// o = sum 2^(m_i - M) o_i / L, lse = (M + log2 L) ln 2.  A row gets 1, 4 or
// 16 warps by its number of splits (one warp per row and four rows per CTA
// for large batches of short contexts, 16 for small batches of long ones).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <atomic>

#include "fa_internal.h"
#include "ptx.cuh"
#include "checks.cuh"

namespace fa {

template <int D>
struct DecodeLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kDecodeBlock * 128;   // 16 tokens x 64 bf16
  static constexpr int kBlockBytes = kChunks * kChunkBytes;  // one KV head of one block
  static constexpr int kStageBytes = 2 * kBlockBytes;        // K then V
  static constexpr int kBar = kDecodeStages * kStageBytes;
  static constexpr int kMisc = kBar + kDecodeStages * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;
};

// Byte offset of element (token, col) of a [16 x D] block staged with
// 128-byte swizzle as D/64 chunks of [16 rows][128 B].
__device__ __forceinline__ uint32_t swz_off(int token, int col) {
  const int chunk = col >> 6;
  const int unit = (col & 63) >> 3;  // 16-byte unit inside the 128-byte row
  return chunk * (kDecodeBlock * 128) + token * 128 + ((unit ^ (token & 7)) << 4);
}

// Keep the bf16 halves of x whose token index is below n_valid.
__device__ __forceinline__ uint32_t keep_tokens(uint32_t x, int tok_lo, int n_valid) {
  const uint32_t lo = (tok_lo < n_valid) ? 0x0000FFFFu : 0u;
  const uint32_t hi = (tok_lo + 1 < n_valid) ? 0xFFFF0000u : 0u;
  return x & (lo | hi);
}

// One warp's pass over a range of keys: the unnormalised O^T accumulator of
// the group's query heads (m16n8 accumulator layout: rows are the head
// dimension, columns the heads), the running maximum of each head (log2
// units) and each lane's share of the row sums.
template <int D, int NT>
struct WarpRange {
  float acc[NT][D / 16][4];
  float mcol[NT][2], lcol[NT][2];
};

constexpr int kRangeOk = 0, kRangeBadBlock = 1, kRangeFailed = 2;

// A converged warp streams keys [t0, t1) (at most kDecodeMaxSplitTokens) of
// sequence b and KV head kvh through its own ring of TMA stages at `smem`
// (DecodeLayout<D>::kBytes, 1024-byte aligned) and leaves its state in st.
// Lane i holds the physical id of logical block t0 / 16 + i in my_blk (-1
// when it could not be read).  Returns kRangeBadBlock (nothing loaded,
// status raised) when a block id of the range is outside the pool,
// kRangeFailed when a wait gave up (copies in flight are drained before it
// returns).
template <int D, int NT>
__device__ __forceinline__ int decode_range(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                            const DecodeParams &p, int b, int kvh, int t0, int t1,
                                            int my_blk, uint8_t *smem, WarpRange<D, NT> &st) {
  using L = DecodeLayout<D>;
  constexpr int S = kDecodeStages;
  constexpr int KC = D / 16;  // 16-wide k chunks of the head dimension
  const int lane = threadIdx.x & 31;
  const int nblk = (t1 - t0 + kDecodeBlock - 1) / kDecodeBlock;  // <= 32
  const int G = p.group;

  const bool bad = lane < nblk && (my_blk < 0 || my_blk >= p.num_blocks);
  const size_t part_row = static_cast<size_t>(b) * p.H + static_cast<size_t>(kvh) * G;
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) raise_status(p.status, FA_DEV_BAD_BLOCK);
    return kRangeBadBlock;
  }

  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBar);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc);

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncwarp();

  auto issue = [&](int st, int phys) {
    uint8_t *dst = smem + st * L::kStageBytes;
    mbar_arrive_expect_tx(&full[st], L::kStageBytes);
#pragma unroll
    for (int c = 0; c < L::kChunks; ++c) {
      tma_load_3d(dst + c * L::kChunkBytes, &tm_k, &full[st], c * 64, kvh, phys * kDecodeBlock);
      tma_load_3d(dst + L::kBlockBytes + c * L::kChunkBytes, &tm_v, &full[st], c * 64, kvh,
                  phys * kDecodeBlock);
    }
  };
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int phys = __shfl_sync(0xffffffffu, my_blk, i);
    if (lane == 0 && i < nblk) issue(i, phys);
  }

  // Q^T fragments (B operand): column n = query head kvh*G + n of the group.
  uint32_t qf[NT][KC][2];
  const int quad = lane & 3;
  const int grp = lane >> 2;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = nt * 8 + grp;
    const bool valid =
        n < G && in_bounds((part_row + n) * D, D, static_cast<size_t>(p.batch) * p.H * D, p.status);
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
        static_cast<const uint16_t *>(p.q) + (part_row + (valid ? n : 0)) * D);
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
      qf[nt][kc][0] = valid ? qrow[(kc * 16 + 2 * quad) >> 1] : 0u;
      qf[nt][kc][1] = valid ? qrow[(kc * 16 + 8 + 2 * quad) >> 1] : 0u;
    }
  }

  float (&acc)[NT][KC][4] = st.acc;
  float (&mcol)[NT][2] = st.mcol;
  float (&lcol)[NT][2] = st.lcol;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < KC; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
    mcol[nt][0] = mcol[nt][1] = -CUDART_INF_F;
    lcol[nt][0] = lcol[nt][1] = 0.f;
  }
  const float sl2 = p.scale_log2;

  // ldmatrix row addresses: lane supplies row (lane & 7) of matrix (lane >> 3).
  const int mi = lane >> 3;
  const int mr = lane & 7;
  // K (non-transposed A operand): matrix mi covers tokens 8*(mi&1).., cols 8*(mi>>1)..
  const int k_tok = mr + 8 * (mi & 1);
  const int k_col = 8 * (mi >> 1);
  // V^T (transposed load): matrix mi covers tokens 8*(mi>>1).., cols 8*(mi&1)..
  const int v_tok = mr + 8 * (mi >> 1);
  const int v_col = 8 * (mi & 1);

  bool ok = true;
  for (int i = 0; i < nblk; ++i) {
    const int st = i % S;
    ok = mbar_wait(&full[st], (i / S) & 1, abort_flag, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const uint32_t kb = smem_u32(smem + st * L::kStageBytes);
    const uint32_t vb = kb + L::kBlockBytes;
    const int n_valid = min(kDecodeBlock, t1 - (t0 + i * kDecodeBlock));

    // S^T = K Q^T
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(kb + swz_off(k_tok, kc * 16 + k_col), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_m16n8k16_bf16(s[nt], a0, a1, a2, a3, qf[nt][kc][0], qf[nt][kc][1]);
    }
    // rows of the accumulator are tokens grp and grp + 8
    if (n_valid < kDecodeBlock) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (grp >= n_valid) s[nt][0] = s[nt][1] = -CUDART_INF_F;
        if (grp + 8 >= n_valid) s[nt][2] = s[nt][3] = -CUDART_INF_F;
      }
    }
    // column-wise (per query head) online softmax
    uint32_t pb0[NT], pb1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pv[4];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float mx = fmaxf(s[nt][cc], s[nt][2 + cc]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(mcol[nt][cc], mx * sl2);
        const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        const float alpha = ex2(mcol[nt][cc] - m_use);
        pv[cc] = ex2(fmaf(s[nt][cc], sl2, -m_use));
        pv[2 + cc] = ex2(fmaf(s[nt][2 + cc], sl2, -m_use));
        lcol[nt][cc] = lcol[nt][cc] * alpha + pv[cc] + pv[2 + cc];
        mcol[nt][cc] = m_new;
#pragma unroll
        for (int mt = 0; mt < KC; ++mt) {
          acc[nt][mt][cc] *= alpha;
          acc[nt][mt][2 + cc] *= alpha;
        }
      }
      pb0[nt] = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));
      pb1[nt] = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));
    }
    // O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < KC; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4_trans(vb + swz_off(v_tok, mt * 16 + v_col), a0, a1, a2, a3);
      if (n_valid < kDecodeBlock) {
        // never let a stale slot past the context reach the accumulator
        a0 = keep_tokens(a0, 2 * quad, n_valid);
        a1 = keep_tokens(a1, 2 * quad, n_valid);
        a2 = keep_tokens(a2, 8 + 2 * quad, n_valid);
        a3 = keep_tokens(a3, 8 + 2 * quad, n_valid);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_m16n8k16_bf16(acc[nt][mt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
    }
    __syncwarp();
    const int nxt = i + S;
    const int phys = __shfl_sync(0xffffffffu, my_blk, nxt & 31);
    if (lane == 0 && nxt < nblk) {
      fence_proxy_async_smem();
      issue(st, phys);
    }
  }

  if (ok) return kRangeOk;
    // drain copies still in flight before the CTA releases its shared memory
    if (lane == 0) {
      for (int i = 0; i < min(nblk, S); ++i) {
        const uint64_t tstart = globaltimer_ns();
        // the last load issued into stage i has phase ((last) / S) & 1
        int last = i;
        while (last + S < nblk) last += S;
        while (!mbar_try_wait(&full[i], (last / S) & 1)) {
          if (globaltimer_ns() - tstart > kWaitLimitNs) break;
        }
      }
    }
    __syncwarp();
  return kRangeFailed;
}

template <int D, int NT>
__global__ void __launch_bounds__(32)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  constexpr int KC = D / 16;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int lane = threadIdx.x;
  pdl_launch_dependents();

  // The block ids of the whole split are read together with the context
  // length (one memory round trip instead of two); ids past the context are
  // not used.
  const int lb0 = split * (p.split_tokens / kDecodeBlock);
  int my_blk = -1;
  if (lane < p.split_tokens / kDecodeBlock && lb0 + lane < p.max_blocks_per_seq) {
    const size_t tidx = static_cast<size_t>(b) * p.max_blocks_per_seq + lb0 + lane;
    if (in_bounds(tidx, 1, static_cast<size_t>(p.batch) * p.max_blocks_per_seq, p.status))
      my_blk = p.block_table[tidx];
  }
  const int ctx = checked_load(p.ctx_lens, b, p.batch, p.status);
  if (ctx < 0 || ctx > p.max_ctx_len || ctx > p.max_blocks_per_seq * kDecodeBlock) {
    if (split == 0 && kvh == 0 && lane == 0) raise_status(p.status, FA_DEV_BAD_CTX);
    return;
  }
  const int t0 = split * p.split_tokens;
  if (t0 >= ctx) return;
  const int t1 = min(ctx, t0 + p.split_tokens);
  const int G = p.group;
  // partial-state rows of the call: [batch, H, max_splits]
  const size_t part_rows = static_cast<size_t>(p.batch) * p.H * p.max_splits;
  const size_t part_row = static_cast<size_t>(b) * p.H + static_cast<size_t>(kvh) * G;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  WarpRange<D, NT> st;
  const int rc = decode_range<D, NT>(tm_k, tm_v, p, b, kvh, t0, t1, my_blk, smem, st);
  if (rc == kRangeBadBlock) {
    // Leave a neutral partial state so that the combine ignores this split.
    for (int g = 0; g < G; ++g) {
      const size_t row = (part_row + g) * p.max_splits + split;
      if (!in_bounds(row, 1, part_rows, p.status)) continue;
      for (int c = lane; c < D; c += 32) p.o_part[row * D + c] = 0.f;
      if (lane == 0) {
        p.ml_part[row * 2 + 0] = -CUDART_INF_F;
        p.ml_part[row * 2 + 1] = 0.f;
      }
    }
    return;
  }
  if (rc != kRangeOk) return;
  // write the partial state of every query head of the group
  const int quad = lane & 3;
  const int grp = lane >> 2;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float lt = st.lcol[nt][cc];
      lt += __shfl_xor_sync(0xffffffffu, lt, 4);
      lt += __shfl_xor_sync(0xffffffffu, lt, 8);
      lt += __shfl_xor_sync(0xffffffffu, lt, 16);
      const int g = nt * 8 + 2 * quad + cc;
      if (g < G) {
        const size_t row = (part_row + g) * p.max_splits + split;
        if (!in_bounds(row, 1, part_rows, p.status)) continue;
        if (grp == 0) {
          p.ml_part[row * 2 + 0] = st.mcol[nt][cc];
          p.ml_part[row * 2 + 1] = lt;
        }
        float *orow = p.o_part + row * D;
#pragma unroll
        for (int mt = 0; mt < KC; ++mt) {
          orow[mt * 16 + grp] = st.acc[nt][mt][cc];
          orow[mt * 16 + 8 + grp] = st.acc[nt][mt][2 + cc];
        }
      }
    }
  }
}

// Warps per merged row: one for rows of at most kCombineFewSplits splits
// (four rows per CTA), kCombineWarps up to kCombineManySplits, and
// kCombineWarpsMany beyond (rows of many short splits: small batches).
constexpr int kCombineFewSplits = 8;
constexpr int kCombineManySplits = 64;
constexpr int kCombineWarpsMany = 16;

template <int W>
constexpr int combine_cta_warps() { return W < 4 ? 4 : W; }

template <int D, int W>
__global__ void __launch_bounds__(32 * combine_cta_warps<W>())
    decode_combine_kernel(const DecodeParams p) {
  // W warps per (sequence, query head) row, R rows per CTA.  The W warps of
  // a row first find M together (thread t of the row reads the maxima of
  // splits t, t + 32 W, ...); then warp w of the row merges splits w, w + W,
  // ..., U of them per memory round trip, and the warps' sums are added
  // through shared memory.  Lane l owns output elements [l E, l E + E).
  constexpr int kWarps = combine_cta_warps<W>();
  constexpr int R = kWarps / W;
  constexpr int E = D / 32;
  constexpr int U = 8;
  __shared__ float s_acc[kWarps][D];
  __shared__ float s_l[kWarps];
  __shared__ float s_m[kWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // this kernel's own (checked-build) index errors go to the device word only
  unsigned int *status = p.dev_status;
  const int wr = warp % W;  // warp within the row
  const int r0 = warp - wr;  // first warp of the row
  const int gw = blockIdx.x * R + warp / W;
  // a CTA's last rows may lie past the end; they still meet the barriers
  const bool row_live = gw < p.batch * p.H;
  const int b = row_live ? gw / p.H : 0;
  int ctx = row_live ? checked_load(p.ctx_lens, b, p.batch, status) : 0;
  if (ctx < 0 || ctx > p.max_ctx_len || ctx > p.max_blocks_per_seq * kDecodeBlock) ctx = 0;
  const int ns = (ctx + p.split_tokens - 1) / p.split_tokens;
  const size_t row0 = static_cast<size_t>(gw) * p.max_splits;
  const size_t part_rows = static_cast<size_t>(p.batch) * p.H * p.max_splits;
  pdl_wait_primary();  // the split grid's partial states are complete from here on
  // The split grid has raised all its status bits: one thread reads them
  // here and publishes them as the call's status when its row is done.
  const bool publisher = blockIdx.x == 0 && threadIdx.x == 0 && p.call != nullptr;
  const unsigned int call_bits = publisher ? call_status_bits(p.call) : 0u;
  // (m, l) of split i of this row (the neutral state if the index fails a
  // check of the checked build)
  auto ml = [&](int i) -> float2 {
    return in_bounds(row0 + i, 1, part_rows, status)
               ? reinterpret_cast<const float2 *>(p.ml_part)[row0 + i]
               : make_float2(-CUDART_INF_F, 0.f);
  };

  float M = -CUDART_INF_F;
  for (int i = wr * 32 + lane; i < ns; i += 32 * W) M = fmaxf(M, ml(i).x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_m[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < W; ++w) M = fmaxf(M, s_m[r0 + w]);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float Lsum = 0.f;
  // Split i adds 2^(m_i - M) (l_i, o_i).  An empty split (m_i = -inf) is
  // passed over by a select, never multiplied in, so whatever its o_i slot
  // holds cannot reach the output.
  if (M != -CUDART_INF_F) {
    auto add = [&](const float2 st, const float (&v)[E]) {
      const bool live = st.x != -CUDART_INF_F;
      const float w = ex2(st.x - M);
      Lsum = live ? fmaf(w, st.y, Lsum) : Lsum;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = live ? fmaf(w, v[e], acc[e]) : acc[e];
    };
    auto load_o = [&](int i, float (&v)[E]) {
      const float *orow = p.o_part + (row0 + i) * D + lane * E;
      if (!in_bounds((row0 + i) * D + lane * E, E, part_rows * D, status)) {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = 0.f;
        return;
      }
      if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(orow);
        v[0] = x.x;
        v[1 % E] = x.y;
        v[2 % E] = x.z;
        v[3 % E] = x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2 *>(orow);
        v[0] = x.x;
        v[1 % E] = x.y;
      }
    };
    int i = wr;
    for (; i + (U - 1) * W < ns; i += U * W) {
      float2 st[U];
      float v[U][E];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        st[u] = ml(i + u * W);
        load_o(i + u * W, v[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) add(st[u], v[u]);
    }
    for (; i < ns; i += W) {
      float v[E];
      load_o(i, v);
      add(ml(i), v);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
  if (lane == 0) s_l[warp] = Lsum;
  __syncthreads();
  if (wr != 0 || !row_live) return;
  Lsum = 0.f;
#pragma unroll
  for (int w = 0; w < W; ++w) Lsum += s_l[r0 + w];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) t += s_acc[r0 + w][lane * E + e];
    acc[e] = t;
  }
  const float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
  uint16_t *dst = static_cast<uint16_t *>(p.out) + static_cast<size_t>(gw) * D + lane * E;
  const bool out_ok = in_bounds(static_cast<size_t>(gw) * D + lane * E, E,
                                static_cast<size_t>(p.batch) * p.H * D, status);
  if (out_ok && E == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1 % E] * inv);
    w.y = pack_bf16x2(acc[2 % E] * inv, acc[3 % E] * inv);
    *reinterpret_cast<uint2 *>(dst) = w;
  } else if (out_ok) {
    *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1 % E] * inv);
  }
  if (lane == 0 && p.lse != nullptr &&
      in_bounds(gw, 1, static_cast<size_t>(p.batch) * p.H, status))
    p.lse[gw] = (Lsum > 0.f) ? (M + __log2f(Lsum)) * 0.69314718055994530942f : -CUDART_INF_F;
  if (publisher) publish_call_status(p.call, call_bits, p.dev_status);
}

// ------------------------------------------------------------------ launch

// The combine grid, launched as a programmatic dependent of the split grid
// on the same stream.
template <int D, int W>
static cudaError_t launch_combine(const DecodeParams &p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(32 * combine_cta_warps<W>());
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, W>, p);
}

template <int D, int NT>
static cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv,
                                   const DecodeParams &p, cudaStream_t stream) {
  using L = DecodeLayout<D>;
  auto kern = decode_split_kernel<D, NT>;
  // The shared-memory attribute is per device: set it once on each device
  // (one bit per device id; ids past 63 set it on every launch).
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit == 0ull || (attr_set.load(std::memory_order_acquire) & bit) == 0ull) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  dim3 grid(p.max_splits, p.Hkv, p.batch);
  kern<<<grid, 32, L::kSmemAlloc, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = p.batch * p.H;
  if (p.max_splits > kCombineManySplits)
    return launch_combine<D, kCombineWarpsMany>(p, rows, stream);
  if (p.max_splits > kCombineFewSplits) return launch_combine<D, kCombineWarps>(p, rows, stream);
  return launch_combine<D, 1>(p, (rows + 3) / 4, stream);
}

cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          int d, cudaStream_t stream) {
  const bool two = p.group > 8;
  if (d == 64) return two ? launch_decode_t<64, 2>(tk, tv, p, stream)
                          : launch_decode_t<64, 1>(tk, tv, p, stream);
  return two ? launch_decode_t<128, 2>(tk, tv, p, stream)
             : launch_decode_t<128, 1>(tk, tv, p, stream);
}

}  // namespace fa
