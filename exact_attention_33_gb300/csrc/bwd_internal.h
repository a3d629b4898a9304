// bwd_internal.h - parameter block and constants of the backward kernels,
// shared by the host glue (fa_api.cu) and backward.cu.  Passed by value.
#pragma once

#include <stdint.h>

#include "fa_internal.h"

namespace fa {

// ----------------------------------------------------------------- backward

constexpr int kBwdThreads = 320;  // 8 elementwise warps + 1 MMA warp + 1 TMA warp
constexpr int kBwdOrderMaxSeqs = 128;  // multiple of 32

struct BwdParams {
  unsigned int *status;   // per-device sticky FA_DEV_* word
  const void *out;        // forward output O, bf16 [B, N, H, d] (packed: [T, H, d])
  const void *dout;       // upstream gradient dO, layout of out
  const float *lse;       // forward log-sum-exp, fp32 [B, H, N] (packed: [H, T]) (natural log)
  float *nlse2;           // workspace: -lse in log2 units, [B, H, Npad]
  float *ndsum;           // workspace: -D = -rowsum(dO * O), [B, H, Npad]
  void *dq, *dk, *dv;     // bf16, layouts of q, k, v
  int B, H, Hkv, group, N;  // packed batches: B sequences of at most N (max_seqlen) rows
  int Npad;               // N rounded up to 128
  int n_tiles;            // Npad / 128
  float scale;            // softmax scale
  float scale_log2;       // scale * log2(e)
  const int32_t *cu_seqlens;  // packed batches only: sequence b is rows [cu[b], cu[b + 1])
  int total_tokens;           // packed batches only: T
  int longest_first;          // packed batches of at most kBwdOrderMaxSeqs sequences: CTAs take
                              // the tiles in longest-first order
  unsigned int *work;         // workspace: work counters of the dQ [0] and dK/dV [1] kernels
                              // (zeroed by the preprocess kernel)
  int num_ctas;               // CTAs of a persistent kernel (the SM count)
};

}  // namespace fa
