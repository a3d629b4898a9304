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
//   warp 9      TMA producer: Q tiles once, then K/V tiles of 128 keys into a
//               ring of shared-memory stages (128-byte swizzle).
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
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

template <int D>
struct PrefillLayout {
  static constexpr int kChunkBytes = 128 * 128;        // 128 rows x 64 bf16 (one swizzle span)
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kPrefillQTiles * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  // q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 1 + 3 * kStages + 7;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;     // base is aligned up to 1024 in-kernel
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kTmemO = 256;
};

// Wait that ignores the abort flag (used only to drain in-flight copies
// before the CTA exits); bounded by the same time limit.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, unsigned int *status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      raise_status(status, FA_DEV_TIMEOUT);
      return;
    }
  }
}

// Loads 32 TMEM columns and waits for them in one asm block, so that no use
// of the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillLayout<D>;
  constexpr int S = L::kStages;

  // ---------------------------------------------------------- work item
  // One CTA per (sequence, 256-row query pair, head); heads vary fastest so
  // that CTAs sharing a KV head run together.  For causal attention the
  // pairs with the most key tiles are launched first.
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int r = lin / p.H;
  int b, pair, seq_start, len;
  if (VARLEN) {
    const int s = r % p.B;
    pair = p.max_pairs - 1 - r / p.B;
    seq_start = p.cu_seqlens[s];
    const int seq_end = p.cu_seqlens[s + 1];
    if (seq_start < 0 || seq_end < seq_start || seq_end > p.total_tokens) {
      if (pair == 0 && h == 0) raise_status(p.status, FA_DEV_BAD_SEQLEN);
      return;
    }
    len = seq_end - seq_start;
    if (len > p.max_pairs * kPrefillRowsPerCta && pair == 0 && h == 0)
      raise_status(p.status, FA_DEV_BAD_SEQLEN);  // longer than max_seqlen: tail not covered
    b = 0;
  } else {
    b = r % p.B;
    pair = CAUSAL ? (p.max_pairs - 1 - r / p.B) : (r / p.B);
    seq_start = 0;
    len = p.N;
  }
  const int row0 = pair * kPrefillRowsPerCta;
  if (row0 >= len) return;  // no padding work: the whole CTA leaves before any set-up

  const int n_kv_all = (len + kPrefillBN - 1) / kPrefillBN;
  int kv_end[kPrefillQTiles];
#pragma unroll
  for (int i = 0; i < kPrefillQTiles; ++i) {
    const int t0 = row0 + i * kPrefillBM;
    if (t0 >= len) {
      kv_end[i] = 0;
    } else {
      kv_end[i] = CAUSAL ? min(n_kv_all, t0 / kPrefillBN + 1) : n_kv_all;
    }
  }
  const int n_kv = max(kv_end[0], kv_end[1]);

  // ---------------------------------------------------------- shared memory
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *v_full = bars + 1 + S;
  uint64_t *kv_empty = bars + 1 + 2 * S;
  uint64_t *s_full = bars + 1 + 3 * S;
  uint64_t *p_full = s_full + 2;
  uint64_t *o_done = p_full + 2;
  uint64_t *drain = o_done + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint8_t *sQ = smem + L::kQ;
  uint8_t *sK = smem + L::kK;
  uint8_t *sV = smem + L::kV;
  const int kvh = h / p.group;

  if (warp == 9) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int nq = (kv_end[1] > 0) ? 2 : 1;
      mbar_arrive_expect_tx(q_full, nq * L::kTileBytes);
      for (int i = 0; i < nq; ++i) {
        const int qrow = seq_start + row0 + i * kPrefillBM;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sQ + i * L::kTileBytes + c * L::kChunkBytes, &tm_q, q_full, c * 64, h,
                      qrow, b);
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        if (j >= S && !mbar_wait(&kv_empty[st], ((j / S) - 1) & 1, abort_flag, p.status)) break;
        const int krow = seq_start + j * kPrefillBN;
        mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sK + st * L::kTileBytes + c * L::kChunkBytes, &tm_k, &k_full[st], c * 64,
                      kvh, krow, b);
        mbar_arrive_expect_tx(&v_full[st], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sV + st * L::kTileBytes + c * L::kChunkBytes, &tm_v, &v_full[st], c * 64,
                      kvh, krow, b);
        issued = j + 1;
      }
      // Never leave copies in flight into shared memory that is about to be
      // released: wait for the last load of every stage.
      mbar_drain(q_full, 0, p.status);
      for (int j = max(0, issued - S); j < issued; ++j) {
        mbar_drain(&k_full[j % S], (j / S) & 1, p.status);
        mbar_drain(&v_full[j % S], (j / S) & 1, p.status);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kPrefillBM, kPrefillBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kPrefillBM, D, false, true);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t k_base = smem_u32(sK);
      const uint32_t v_base = smem_u32(sV);

      auto issue_s = [&](int i, int st) {
        const uint32_t d_t = tmem + i * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(q_base + i * L::kTileBytes + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(k_base + st * L::kTileBytes + off, 16, 1024);
          mma_ss(d_t, a, bd, kIdescS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[i]);
      };
      auto issue_o = [&](int i, int st, int j) {
        const uint32_t d_t = tmem + L::kTmemO + i * D;
        const uint32_t p_t = tmem + i * 128;
#pragma unroll
        for (int kk = 0; kk < kPrefillBN / 16; ++kk) {
          const uint64_t bd =
              sdesc_sw128(v_base + st * L::kTileBytes + kk * 2048, L::kChunkBytes, 1024);
          mma_ts(d_t, p_t + kk * 8, bd, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&o_done[i]);
      };

      bool ok = mbar_wait(q_full, 0, abort_flag, p.status) && mbar_wait(&k_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < 2; ++i)
          if (kv_end[i] > 0) issue_s(i, 0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % S;
        const int st1 = (j + 1) % S;
        bool k_next = false;
        if (!mbar_wait(&v_full[st], (j / S) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        for (int i = 0; i < 2 && ok; ++i) {
          if (j < kv_end[i]) {
            if (!mbar_wait(&p_full[i], j & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_o(i, st, j);
          }
          if (j + 1 < kv_end[i]) {
            if (!k_next) {
              if (!mbar_wait(&k_full[st1], ((j + 1) / S) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_next = true;
            }
            issue_s(i, st1);
          }
        }
        mma_commit(&kv_empty[st]);
      }
      // Everything this thread issued must finish before TMEM is released.
      mma_commit(drain);
      mbar_drain(drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------------ softmax warpgroups
    const int i = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + i * 128 + lane_off;
    const uint32_t tO = tmem + L::kTmemO + i * D + lane_off;
    const int qi = row0 + i * kPrefillBM + row;  // query row within the sequence
    const int my_end = kv_end[i];
    const float sl2 = p.scale_log2;
    float m = -CUDART_INF_F;  // running max, log2 units
    float l = 0.f;            // running sum relative to m
    bool ok = true;
    const int limit = CAUSAL ? min(len, qi + 1) : len;  // keys [0, limit) are visible

    for (int j = 0; j < my_end; ++j) {
      ok = mbar_wait(&s_full[i], j & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();

      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32_wait(tS + c * 32, rr);
#pragma unroll
        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(rr[t]);
      }
      const int nvis = limit - j * kPrefillBN;
      if (__any_sync(0xffffffffu, nvis < kPrefillBN)) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= nvis) s[c] = -CUDART_INF_F;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < 128; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m, mx * sl2);
      // NaN guard ("exp(-inf - -inf) is NaN"): a row that has seen no
      // visible key yet keeps a finite reference of 0.
      const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);
      const float neg = -m_use;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2(fmaf(s[2 * c], sl2, neg));
        const float p1 = ex2(fmaf(s[2 * c + 1], sl2, neg));
        rs0 += p0;
        rs1 += p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + (rs0 + rs1);
      {
        uint32_t lo[32], hi[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          lo[c] = pk[c];
          hi[c] = pk[32 + c];
        }
        tmem_st32(tS, lo);
        tmem_st32(tS + 32, hi);
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + c * 32, o);
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[i]);
      m = m_new;
    }

    // ---------------------------------------------------- epilogue
    if (ok && my_end > 0) {
      ok = mbar_wait(&o_done[i], (my_end - 1) & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const bool live = qi < len;
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        size_t out_row;
        if (VARLEN)
          out_row = static_cast<size_t>(seq_start + qi);
        else
          out_row = static_cast<size_t>(b) * p.N + qi;
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) +
                                               ((out_row * p.H + h) * D) * 2);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + c * 32, o);
          if (live) {
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
        if (live && p.lse != nullptr) {
          const float lse =
              (l > 0.f) ? (m + __log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
          if (VARLEN)
            p.lse[static_cast<size_t>(h) * p.total_tokens + seq_start + qi] = lse;
          else
            p.lse[(static_cast<size_t>(b) * p.H + h) * p.N + qi] = lse;
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ------------------------------------------------------------------ launch

template <int D, bool CAUSAL, bool VARLEN>
static cudaError_t launch_prefill_t(const CUtensorMap &tq, const CUtensorMap &tk,
                                    const CUtensorMap &tv, const PrefillParams &p, int grid,
                                    cudaStream_t stream) {
  using L = PrefillLayout<D>;
  auto kern = prefill_kernel<D, CAUSAL, VARLEN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kPrefillThreads, L::kSmemAlloc, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const PrefillParams &p, int d, bool causal, bool varlen, int grid,
                           cudaStream_t stream) {
  if (d == 64) {
    if (varlen)
      return causal ? launch_prefill_t<64, true, true>(tq, tk, tv, p, grid, stream)
                    : launch_prefill_t<64, false, true>(tq, tk, tv, p, grid, stream);
    return causal ? launch_prefill_t<64, true, false>(tq, tk, tv, p, grid, stream)
                  : launch_prefill_t<64, false, false>(tq, tk, tv, p, grid, stream);
  }
  if (varlen)
    return causal ? launch_prefill_t<128, true, true>(tq, tk, tv, p, grid, stream)
                  : launch_prefill_t<128, false, true>(tq, tk, tv, p, grid, stream);
  return causal ? launch_prefill_t<128, true, false>(tq, tk, tv, p, grid, stream)
                : launch_prefill_t<128, false, false>(tq, tk, tv, p, grid, stream);
}

}  // namespace fa
