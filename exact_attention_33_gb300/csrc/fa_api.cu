// fa_api.cu - the C ABI of libfa.so: argument validation, TMA tensor-map
// construction and kernel dispatch.  The host side keeps the strides, dtypes,
// masking mode and sequence layout of every call and hands the kernels a
// plain parameter block (the bridge described in "How the Repo Connects
// Python to Bare-Metal CUDA" of the explainer article on the FlashAttention
// repository); nothing here allocates device memory or synchronises.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "bwd_internal.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

__device__ unsigned int g_status = 0;

cudaError_t launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const CUtensorMap &tv1, const CUtensorMap &to, const PrefillParams &p,
                           int d, bool causal, int kind, int grid, cudaStream_t stream,
                           int qtiles = 2);
cudaError_t launch_prefill_split_combine(const PrefillParams &p, int d, cudaStream_t stream);
cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                       const CUtensorMap &tv, const BwdParams &p, int d, bool causal,
                       cudaStream_t stream);
cudaError_t launch_prefill_fp8(const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, const CUtensorMap &to,
                               const PrefillParams &p, bool causal, int grid,
                               cudaStream_t stream, int kind, int d);
cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          int d, cudaStream_t stream);
cudaError_t launch_call_status(CallStatus *call, unsigned int *dev, cudaStream_t stream);

namespace {

constexpr float kLog2e = 1.4426950408889634f;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tensor [outer][rows][heads][d] (d innermost) of bf16 (or one-byte, or
// fp32) elements as a 4-D TMA map with dims {d, heads, rows, outer}; each
// copy moves a box of one swizzled row of swz_bytes per (head, row): {64, 1,
// box_rows, 1} bf16 values with the 128-byte swizzle, or, for e4m3 rows of
// d = 64, {64, 1, box_rows, 1} bytes with the 64-byte swizzle.
// Out-of-range rows read as zero and are not stored.
int make_map(CUtensorMap *map, const void *base, int d, int heads, long long rows,
             long long outer, int box_rows, int elem_bytes = 2, int swz_bytes = 128) {
  auto fn = encode_fn();
  if (fn == nullptr) return FA_ERR_CUDA;
  const cuuint64_t eb = static_cast<cuuint64_t>(elem_bytes);
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * eb,
                                 static_cast<cuuint64_t>(heads) * d * eb,
                                 static_cast<cuuint64_t>(rows) * heads * d * eb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(swz_bytes / elem_bytes), 1,
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(map, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Swizzled row bytes of the prefill kernels for e4m3 rows of d values.
int fp8_swz(int d) { return d < 128 ? d : 128; }

// Paged pool [num_blocks * block_size tokens][Hkv][d] as a 3-D map; each copy
// moves {64, 1, box_rows} (a whole 16-token block, or one token row).
int make_pool_map(CUtensorMap *map, const void *base, int d, int heads, long long tokens,
                  int box_rows = kDecodeBlock) {
  auto fn = encode_fn();
  if (fn == nullptr) return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(heads) * d * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

// Device address of the sticky status word of the current device (looked up
// once per device).
unsigned int *status_ptr() {
  constexpr int kMaxDev = 64;
  static unsigned int *ptrs[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int *>(p);
  }
  return ptrs[dev];
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Keys per split of the decode kernel.  Large splits keep the partial-state
// traffic small; the split shrinks (down to 64 keys) while the number of
// (sequence, KV head, split) work items would not fill kDecodeWaveCtas split
// CTAs per SM (about two waves of seven resident CTAs).
#ifndef FA_DECODE_WAVE_CTAS
#define FA_DECODE_WAVE_CTAS 14
#endif
constexpr int kDecodeWaveCtas = FA_DECODE_WAVE_CTAS;
int decode_split_tokens(int batch, int Hkv, int max_ctx_len) {
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  const long long want = static_cast<long long>(kDecodeWaveCtas) * sms;
  int split = kDecodeMaxSplitTokens;
  while (split > 64) {
    const long long items = static_cast<long long>(batch) * Hkv *
                            ((static_cast<long long>(max_ctx_len) + split - 1) / split);
    if (items >= want) break;
    split >>= 1;
  }
  return split;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Context lengths above this are refused (the split arithmetic stays in int).
constexpr int kMaxCtxLen = 0x7fffffff - kDecodeMaxSplitTokens;

// Heads per group of the prefill CTA order: the largest divisor of H that is
// at most 8 (consecutive heads, so GQA heads sharing a KV head stay together).
int prefill_head_group(int H) {
  for (int g = 8; g > 1; --g)
    if (H % g == 0) return g;
  return 1;
}

// Splits of the split-KV prefill: about 1.7 CTAs per SM (rounded down), at
// most 16 splits and at most one split per key tile.  Every extra split costs
// an fp32 partial tile per query tile and its share of the combine; on
// B1 H4 N8192 causal (128 work items on 152 SMs) 2 splits ran at 924 TFLOP/s
// against 796 for 3 and 640 unsplit, and from 256 work items up the unsplit
// kernel was fastest.
int prefill_num_splits(int B, int H, int N, int requested) {
  const long long pairs = (N + kPrefillRowsPerCta - 1) / kPrefillRowsPerCta;
  const int tiles = (N + kPrefillBN - 1) / kPrefillBN;
  int s = requested;
  if (s <= 0) {
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    const long long base = std::max(1LL, pairs * B * H);
    s = static_cast<int>(std::min(16LL, (17LL * sms) / (10LL * base)));
  }
  return std::max(1, std::min({s, 16, std::max(1, tiles)}));
}

struct SplitWs {
  int splits;
  size_t o_bytes, ml_bytes;
};

// Split-KV workspace: control block, fp32 partial o tiles, (m, l, l_exact).
SplitWs split_ws(int B, int H, int N, int d, int requested) {
  SplitWs w;
  w.splits = prefill_num_splits(B, H, N, requested);
  const size_t rows = static_cast<size_t>(w.splits) * B * N * H;
  w.o_bytes = round_up(rows * d * sizeof(float), 256);
  w.ml_bytes = round_up(rows * 4 * sizeof(float), 256);
  return w;
}

size_t split_ws_bytes(const SplitWs &w) { return FA_WORKSPACE_HEADER_BYTES + w.o_bytes + w.ml_bytes; }

struct DecodeWs {
  int split_tokens;
  int max_splits;
  size_t o_bytes;
  size_t ml_bytes;
};

// Decode workspace: control block, fp32 partial o rows, (m, l) pairs.
DecodeWs decode_ws(int batch, int H, int Hkv, int d, int max_ctx_len) {
  DecodeWs w;
  w.split_tokens = decode_split_tokens(batch, Hkv, max_ctx_len);
  w.max_splits = static_cast<int>(std::max(
      1LL, (static_cast<long long>(max_ctx_len) + w.split_tokens - 1) / w.split_tokens));
  const size_t rows = static_cast<size_t>(batch) * H * w.max_splits;
  w.o_bytes = round_up(rows * d * sizeof(float), 256);
  w.ml_bytes = round_up(rows * 2 * sizeof(float), 256);
  return w;
}

// Waits, through the same bounded mbar_wait that every pipeline uses, on an
// mbarrier that nothing arrives at; the wait gives up after kWaitLimitNs and
// raises FA_DEV_TIMEOUT.  Lets the failure path be tested without faulting.
__global__ void wait_timeout_selftest_kernel(unsigned int *status, int *result) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0, &abort_flag, status);
  if (threadIdx.x == 0) *result = ok ? 1 : 0;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int fa_device_status(unsigned int *status, int clear) {
  if (status == nullptr) return FA_ERR_INVALID_ARG;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  *status = v;
  if (clear) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_status, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_last_device_status(const void *workspace) {
  if (workspace == nullptr || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
  unsigned int v = 0;
  const void *src = static_cast<const uint8_t *>(workspace) + offsetof(CallStatus, last);
  cudaError_t e = cudaMemcpyAsync(&v, src, sizeof(v), cudaMemcpyDeviceToHost, cudaStreamPerThread);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamPerThread);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return static_cast<int>(v & 0x7fffffffu);
}

int fa_selftest_wait_timeout(int *wait_result, fa_stream_t stream) {
  if (wait_result == nullptr) return FA_ERR_INVALID_ARG;
  unsigned int *st = status_ptr();
  if (st == nullptr) return FA_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(st,
                                                                                   wait_result);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Dense prefill; `call` (or null) is the control block of a split-KV
// workspace whose call runs this kernel alone.
static int fwd_dense(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                     int H, int Hkv, int N, int d, float scale, int causal, fa_stream_t stream,
                     CallStatus *call) {
  if (!q || !k || !v || !out) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return FA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || H < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || N == 0) return FA_OK;
  // With an even GQA group a CTA holds two query heads of one KV group over
  // the same 128 rows (both tiles share every K/V stage and key tile);
  // otherwise two consecutive 128-row tiles of one head.
  const bool head_pairs = (H / Hkv) % 2 == 0;
  const int rows = head_pairs ? kPrefillBM : kPrefillRowsPerCta;  // rows per work item
  const long long pairs = (N + rows - 1) / rows;
  const long long grid = pairs * B * (head_pairs ? H / 2 : H);
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * H * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;

  CUtensorMap tq, tk, tv, to;
  int rc = make_map(&tq, q, d, H, N, B, kPrefillBM);
  if (rc == FA_OK) rc = make_map(&tk, k, d, Hkv, N, B, kPrefillBN);
  if (rc == FA_OK) rc = make_map(&tv, v, d, Hkv, N, B, kPrefillBN);
  if (rc == FA_OK) rc = make_map(&to, out, d, H, N, B, kPrefillBM);
  if (rc != FA_OK) return rc;

  PrefillParams p{};
  p.dev_status = status_ptr();
  if (p.dev_status == nullptr) return FA_ERR_CUDA;
  // a split-KV call running this kernel alone raises into its workspace
  p.status = call != nullptr ? &call->acc : p.dev_status;
  p.out = out;
  p.lse = lse;
  p.cu_seqlens = nullptr;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.head_group = head_pairs ? 2 * prefill_head_group(H / 2) : prefill_head_group(H);
  p.N = N;
  p.max_pairs = static_cast<int>(pairs);
  p.total_tokens = 0;
  p.scale_log2 = scale * kLog2e;
  p.v_descale = 1.f;
  p.causal = causal;
  p.prefetch_ahead = std::max(0, sm_count());  // one CTA per SM
  cudaError_t e = launch_prefill(tq, tk, tv, tv, to, p, d, causal != 0,
                                 head_pairs ? kKindDenseHeads : kKindDense,
                                 static_cast<int>(grid), reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess && call != nullptr)
    e = launch_call_status(call, p.dev_status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
           int Hkv, int N, int d, float scale, int causal, fa_stream_t stream) {
  return fwd_dense(q, k, v, out, lse, B, H, Hkv, N, d, scale, causal, stream, nullptr);
}

// Packed varlen prefill, bf16 or (fp8) e4m3 codes with per-tensor descales.
static int fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                      const int32_t *cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                      int H, int Hkv, int d, float scale, int causal, fa_stream_t stream, bool fp8,
                      float q_descale, float k_descale, float v_descale) {
  if (!q || !k || !v || !out || !cu_seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return FA_ERR_INVALID_ARG;
  if (!aligned(cu_seqlens, 4) || (lse && !aligned(lse, 4))) return FA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return FA_ERR_INVALID_ARG;
  if (H < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale) || !scale_ok(q_descale) || !scale_ok(k_descale) || !scale_ok(v_descale))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return FA_OK;
  if (max_seqlen > total_tokens) max_seqlen = total_tokens;
  // Work layouts of a packed batch.  With an even GQA group a CTA pairs two
  // query heads of one KV group over the same 128 rows: the two tiles share
  // every K/V stage and have the same key tiles (3-5% faster than the other
  // layouts at every length measured).  Otherwise batches of short sequences
  // (under 4096 rows on average) run one query tile per CTA, two CTAs per SM,
  // and longer sequences pair two consecutive 128-row tiles of one head (the
  // fp8 kernel has the two-tile layouts only).
  constexpr int kRowsOne = 0, kRowPairs = 1, kHeadPairs = 2;
  const bool short_seqs = !fp8 && static_cast<long long>(total_tokens) < 4096LL * num_seqs;
  const int layout = ((H / Hkv) % 2 == 0) ? kHeadPairs : (short_seqs ? kRowsOne : kRowPairs);
  const int qtiles = layout == kRowsOne ? 1 : 2;
  const int rows = layout == kRowPairs ? 2 * kPrefillBM : kPrefillBM;  // rows per work item
  const int slots = layout == kHeadPairs ? H / 2 : H;                 // head slots per row block
  const long long pairs = (max_seqlen + rows - 1) / rows;
  long long grid = pairs * num_seqs * slots;
  // Padding-free order: sum over sequences of ceil(len / rows) is at most
  // ceil(T / rows) + num_seqs, so that many items per head slot cover every row.
  const bool compact = num_seqs <= kVarlenCompactMaxSeqs;
  if (compact)
    grid = std::min(grid,
                    ((total_tokens + rows - 1) / rows + static_cast<long long>(num_seqs)) * slots);
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(total_tokens) * H * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;

  const int eb = fp8 ? 1 : 2;               // bytes per q, k, v element
  const int swz = fp8 ? fp8_swz(d) : 128;   // swizzled row bytes
  CUtensorMap tq, tk, tv, to;
  int rc = make_map(&tq, q, d, H, total_tokens, 1, kPrefillBM, eb, swz);
  if (rc == FA_OK) rc = make_map(&tk, k, d, Hkv, total_tokens, 1, kPrefillBN, eb, swz);
  if (rc == FA_OK) rc = make_map(&tv, v, d, Hkv, total_tokens, 1, kPrefillBN, eb, swz);
  if (rc == FA_OK) rc = make_map(&to, out, d, H, total_tokens, 1, kPrefillBM);
  if (rc != FA_OK) return rc;

  PrefillParams p{};
  p.status = status_ptr();
  if (p.status == nullptr) return FA_ERR_CUDA;
  p.out = out;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.B = num_seqs;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  // heads per CTA-ordering group; a whole number of head pairs for that layout
  p.head_group = layout == kHeadPairs ? 2 * prefill_head_group(H / 2) : prefill_head_group(H);
  p.N = total_tokens;
  p.max_pairs = static_cast<int>(pairs);
  p.compact = compact ? 1 : 0;
  p.total_tokens = total_tokens;
  p.scale_log2 = scale * q_descale * k_descale * kLog2e;
  p.v_descale = v_descale;
  p.causal = causal;
  p.prefetch_ahead = std::max(0, sm_count()) * (qtiles == 1 ? 2 : 1);  // CTAs resident at once
  const int kind = layout == kHeadPairs ? kKindVarlenHeads : kKindVarlen;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = fp8 ? launch_prefill_fp8(tq, tk, tv, to, p, causal != 0, static_cast<int>(grid), st,
                                           kind, d)
                      : launch_prefill(tq, tk, tv, tv, to, p, d, causal != 0, kind,
                                       static_cast<int>(grid), st, qtiles);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                  const int32_t *cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                  int H, int Hkv, int d, float scale, int causal, fa_stream_t stream) {
  return fwd_varlen(q, k, v, out, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, Hkv, d,
                    scale, causal, stream, false, 1.f, 1.f, 1.f);
}

int fa_fwd_varlen_fp8(const void *q, const void *k, const void *v, void *out, float *lse,
                      const int32_t *cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                      int H, int Hkv, int d, float scale, float q_descale, float k_descale,
                      float v_descale, int causal, fa_stream_t stream) {
  return fwd_varlen(q, k, v, out, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, Hkv, d,
                    scale, causal, stream, true, q_descale, k_descale, v_descale);
}

int fa_fwd_fp8(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
               int Hkv, int N, int d, float scale, float q_descale, float k_descale,
               float v_descale, int causal, fa_stream_t stream) {
  if (!q || !k || !v || !out) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return FA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || H < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale) || !scale_ok(q_descale) || !scale_ok(k_descale) ||
      !scale_ok(v_descale))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || N == 0) return FA_OK;
  const long long pairs = (N + kPrefillRowsPerCta - 1) / kPrefillRowsPerCta;
  const long long grid = pairs * B * H;
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * H * d >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv, to;
  int rc = make_map(&tq, q, d, H, N, B, kPrefillBM, 1, fp8_swz(d));
  if (rc == FA_OK) rc = make_map(&tk, k, d, Hkv, N, B, kPrefillBN, 1, fp8_swz(d));
  if (rc == FA_OK) rc = make_map(&tv, v, d, Hkv, N, B, kPrefillBN, 1, fp8_swz(d));
  if (rc == FA_OK) rc = make_map(&to, out, d, H, N, B, kPrefillBM);
  if (rc != FA_OK) return rc;
  PrefillParams p{};
  p.status = status_ptr();
  if (p.status == nullptr) return FA_ERR_CUDA;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.head_group = prefill_head_group(H);
  p.N = N;
  p.max_pairs = static_cast<int>(pairs);
  p.scale_log2 = scale * q_descale * k_descale * kLog2e;
  p.v_descale = v_descale;
  p.causal = causal;
  p.prefetch_ahead = std::max(0, sm_count());
  cudaError_t e = launch_prefill_fp8(tq, tk, tv, to, p, causal != 0, static_cast<int>(grid),
                                     reinterpret_cast<cudaStream_t>(stream), kKindDense, d);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Backward workspace: -lse2 and -D vectors ([B, H, Npad] fp32 each), then a
// 256-byte block holding the work counters of the persistent kernels.
constexpr size_t kBwdCounterBytes = 256;

size_t fa_bwd_workspace_size(int B, int H, int N) {
  if (B <= 0 || H <= 0 || N <= 0) return 0;
  const size_t npad = (static_cast<size_t>(N) + 127) / 128 * 128;
  return 2 * static_cast<size_t>(B) * H * npad * sizeof(float) + kBwdCounterBytes;
}

int fa_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int N, int d,
           float scale, int causal, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  for (const void *ptr : {q, k, v, out, dout, static_cast<const void *>(dq),
                          static_cast<const void *>(dk), static_cast<const void *>(dv)})
    if (!aligned(ptr, 16)) return FA_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return FA_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || H < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || N == 0) return FA_OK;
  const size_t need = fa_bwd_workspace_size(B, H, N);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return FA_ERR_WORKSPACE;
  const long long n_tiles = (N + 127) / 128;
  if (n_tiles * B * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * H * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;

  CUtensorMap tq, tdo, tk, tv;
  int rc = make_map(&tq, q, d, H, N, B, 128);
  if (rc == FA_OK) rc = make_map(&tdo, dout, d, H, N, B, 128);
  if (rc == FA_OK) rc = make_map(&tk, k, d, Hkv, N, B, 128);
  if (rc == FA_OK) rc = make_map(&tv, v, d, Hkv, N, B, 128);
  if (rc != FA_OK) return rc;

  BwdParams p{};
  p.status = status_ptr();
  if (p.status == nullptr) return FA_ERR_CUDA;
  p.out = out;
  p.dout = dout;
  p.lse = lse;
  p.n_tiles = static_cast<int>(n_tiles);
  p.Npad = p.n_tiles * 128;
  p.nlse2 = static_cast<float *>(workspace);
  p.ndsum = p.nlse2 + static_cast<size_t>(B) * H * p.Npad;
  p.work = reinterpret_cast<unsigned int *>(p.ndsum + static_cast<size_t>(B) * H * p.Npad);
  p.num_ctas = std::max(1, sm_count());
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.N = N;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  cudaError_t e = launch_bwd(tq, tdo, tk, tv, p, d, causal != 0,
                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *out, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, const int32_t *cu_seqlens,
                  int num_seqs, int total_tokens, int max_seqlen, int H, int Hkv, int d,
                  float scale, int causal, void *workspace, size_t workspace_bytes,
                  fa_stream_t stream) {
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !cu_seqlens)
    return FA_ERR_INVALID_ARG;
  for (const void *ptr : {q, k, v, out, dout, static_cast<const void *>(dq),
                          static_cast<const void *>(dk), static_cast<const void *>(dv)})
    if (!aligned(ptr, 16)) return FA_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(cu_seqlens, 4)) return FA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return FA_ERR_INVALID_ARG;
  if (H < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return FA_OK;
  const int n_max = std::min(max_seqlen, total_tokens);
  const size_t need = fa_bwd_workspace_size(num_seqs, H, n_max);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return FA_ERR_WORKSPACE;
  const long long n_tiles = (n_max + 127) / 128;
  if (n_tiles * num_seqs * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(total_tokens) * H * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;

  // the packed tensors as one batch element of total_tokens rows; each CTA
  // offsets its row coordinates by its sequence's first row
  CUtensorMap tq, tdo, tk, tv;
  int rc = make_map(&tq, q, d, H, total_tokens, 1, 128);
  if (rc == FA_OK) rc = make_map(&tdo, dout, d, H, total_tokens, 1, 128);
  if (rc == FA_OK) rc = make_map(&tk, k, d, Hkv, total_tokens, 1, 128);
  if (rc == FA_OK) rc = make_map(&tv, v, d, Hkv, total_tokens, 1, 128);
  if (rc != FA_OK) return rc;

  BwdParams p{};
  p.status = status_ptr();
  if (p.status == nullptr) return FA_ERR_CUDA;
  p.out = out;
  p.dout = dout;
  p.lse = lse;
  p.n_tiles = static_cast<int>(n_tiles);
  p.Npad = p.n_tiles * 128;
  p.nlse2 = static_cast<float *>(workspace);
  p.ndsum = p.nlse2 + static_cast<size_t>(num_seqs) * H * p.Npad;
  p.work = reinterpret_cast<unsigned int *>(p.ndsum + static_cast<size_t>(num_seqs) * H * p.Npad);
  p.num_ctas = std::max(1, sm_count());
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = num_seqs;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.N = n_max;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.cu_seqlens = cu_seqlens;
  p.total_tokens = total_tokens;
  p.longest_first = num_seqs <= kBwdOrderMaxSeqs;
  cudaError_t e = launch_bwd(tq, tdo, tk, tv, p, d, causal != 0,
                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits) {
  if (B < 0 || H < 1 || N < 0 || num_splits < 0 || (d != 64 && d != 128)) return 0;
  return split_ws_bytes(split_ws(B, H, N, d, num_splits));
}

int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                   int H, int Hkv, int N, int d, float scale, int causal, int num_splits,
                   void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!q || !k || !v || !out) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return FA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || num_splits < 0)
    return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || N == 0) return FA_OK;
  const SplitWs w = split_ws(B, H, N, d, num_splits);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < split_ws_bytes(w))
    return FA_ERR_WORKSPACE;
  CallStatus *call = static_cast<CallStatus *>(workspace);
  uint8_t *parts = static_cast<uint8_t *>(workspace) + FA_WORKSPACE_HEADER_BYTES;
  // one split: the plain kernel writes the result directly
  if (w.splits == 1)
    return fwd_dense(q, k, v, out, lse, B, H, Hkv, N, d, scale, causal, stream, call);
  const long long pairs = (N + kPrefillRowsPerCta - 1) / kPrefillRowsPerCta;
  const long long grid = pairs * B * H * w.splits;
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * H * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;

  // The split kernel stores its fp32 partial O tiles, [split][B][N][H][d],
  // through this map: (split, batch) is the outer coordinate.
  CUtensorMap tq, tk, tv, to_part;
  int rc = make_map(&tq, q, d, H, N, B, kPrefillBM);
  if (rc == FA_OK) rc = make_map(&tk, k, d, Hkv, N, B, kPrefillBN);
  if (rc == FA_OK) rc = make_map(&tv, v, d, Hkv, N, B, kPrefillBN);
  if (rc == FA_OK)
    rc = make_map(&to_part, parts, d, H, N, static_cast<long long>(w.splits) * B,
                  kPrefillBM, 4);
  if (rc != FA_OK) return rc;

  PrefillParams p{};
  p.status = status_ptr();
  if (p.status == nullptr) return FA_ERR_CUDA;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.head_group = prefill_head_group(H);
  p.N = N;
  p.max_pairs = static_cast<int>(pairs);
  p.scale_log2 = scale * kLog2e;
  p.v_descale = 1.f;
  p.causal = causal;
  p.num_splits = w.splits;
  p.dev_status = p.status;
  p.status = &call->acc;
  p.call = call;
  p.o_part = reinterpret_cast<float *>(parts);
  p.ml_part = reinterpret_cast<float *>(parts + w.o_bytes);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_prefill(tq, tk, tv, tv, to_part, p, d, causal != 0, kKindDenseSplit,
                                 static_cast<int>(grid), st);
  if (e == cudaSuccess) e = launch_prefill_split_combine(p, d, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_paged(const void *q, const void *k_pool, const void *v_pool,
                 const int32_t *block_table, int max_blocks_per_seq, const int32_t *ctx_lens,
                 const int32_t *cu_seqlens_q, int batch, int total_q, int max_seqlen_q,
                 int max_ctx_len, int H, int Hkv, int d, int block_size, int num_blocks,
                 float scale, int causal, void *out, float *lse, fa_stream_t stream) {
  if (!q || !k_pool || !v_pool || !block_table || !ctx_lens || !cu_seqlens_q || !out)
    return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16))
    return FA_ERR_INVALID_ARG;
  if (!aligned(block_table, 4) || !aligned(ctx_lens, 4) || !aligned(cu_seqlens_q, 4) ||
      (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || max_ctx_len < 0 || H < 1 || Hkv < 1 ||
      H % Hkv != 0 || num_blocks < 1 || max_blocks_per_seq < 1)
    return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (block_size != kDecodeBlock) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size < max_ctx_len)
    return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (max_seqlen_q > total_q) max_seqlen_q = total_q;
  // with an even GQA group, two query heads of one KV group per CTA (as in fa_fwd)
  const bool head_pairs = (H / Hkv) % 2 == 0;
  const int rows = head_pairs ? kPrefillBM : kPrefillRowsPerCta;  // query rows per work item
  const long long pairs = (max_seqlen_q + rows - 1) / rows;
  const long long grid = pairs * batch * (head_pairs ? H / 2 : H);
  if (grid > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(total_q) * H * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;

  CUtensorMap tq, tk, tv, tv1, to;
  const long long tokens = static_cast<long long>(num_blocks) * block_size;
  int rc = make_map(&tq, q, d, H, total_q, 1, kPrefillBM);
  if (rc == FA_OK) rc = make_map(&to, out, d, H, total_q, 1, kPrefillBM);
  if (rc == FA_OK) rc = make_pool_map(&tk, k_pool, d, Hkv, tokens);
  if (rc == FA_OK) rc = make_pool_map(&tv, v_pool, d, Hkv, tokens);
  if (rc == FA_OK) rc = make_pool_map(&tv1, v_pool, d, Hkv, tokens, 1);
  if (rc != FA_OK) return rc;

  PrefillParams p{};
  p.status = status_ptr();
  if (p.status == nullptr) return FA_ERR_CUDA;
  p.out = out;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens_q;
  p.B = batch;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.head_group = head_pairs ? 2 * prefill_head_group(H / 2) : prefill_head_group(H);
  p.N = total_q;
  p.max_pairs = static_cast<int>(pairs);
  p.total_tokens = total_q;
  p.scale_log2 = scale * kLog2e;
  p.v_descale = 1.f;
  p.causal = causal;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_ctx_len = max_ctx_len;
  p.num_blocks = num_blocks;
  cudaError_t e = launch_prefill(tq, tk, tv, tv1, to, p, d, causal != 0,
                                 head_pairs ? kKindPagedHeads : kKindPaged,
                                 static_cast<int>(grid), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_decode_workspace_size(int batch, int H, int Hkv, int d, int max_ctx_len,
                                int block_size) {
  if (batch < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || max_ctx_len < 0) return 0;
  if ((d != 64 && d != 128) || block_size != kDecodeBlock) return 0;
  if (max_ctx_len > kMaxCtxLen) return 0;
  const DecodeWs w = decode_ws(batch, H, Hkv, d, max_ctx_len);
  return FA_WORKSPACE_HEADER_BYTES + w.o_bytes + w.ml_bytes;
}

int fa_decode_paged(const void *q, const void *k_pool, const void *v_pool,
                    const int32_t *block_table, int max_blocks_per_seq, const int32_t *ctx_lens,
                    int max_ctx_len, int batch, int H, int Hkv, int d, int block_size,
                    int num_blocks, float scale, void *out, float *lse, void *workspace,
                    size_t workspace_bytes, fa_stream_t stream) {
  if (!q || !k_pool || !v_pool || !block_table || !ctx_lens || !out) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16))
    return FA_ERR_INVALID_ARG;
  if (!aligned(block_table, 4) || !aligned(ctx_lens, 4) || (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  if (batch < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || num_blocks < 1 ||
      max_blocks_per_seq < 1 || max_ctx_len < 0)
    return FA_ERR_INVALID_ARG;
  if (max_ctx_len > kMaxCtxLen) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (block_size != kDecodeBlock) return FA_ERR_UNSUPPORTED;
  if (H / Hkv > 16) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size < max_ctx_len)
    return FA_ERR_INVALID_ARG;
  if (batch > 65535 || Hkv > 65535) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (batch == 0) return FA_OK;
  const DecodeWs w = decode_ws(batch, H, Hkv, d, max_ctx_len);
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < FA_WORKSPACE_HEADER_BYTES + w.o_bytes + w.ml_bytes)
    return FA_ERR_WORKSPACE;
  CallStatus *call = static_cast<CallStatus *>(workspace);
  uint8_t *parts = static_cast<uint8_t *>(workspace) + FA_WORKSPACE_HEADER_BYTES;

  CUtensorMap tk, tv;
  const long long tokens = static_cast<long long>(num_blocks) * block_size;
  int rc = make_pool_map(&tk, k_pool, d, Hkv, tokens);
  if (rc == FA_OK) rc = make_pool_map(&tv, v_pool, d, Hkv, tokens);
  if (rc != FA_OK) return rc;

  DecodeParams p{};
  p.dev_status = status_ptr();
  if (p.dev_status == nullptr) return FA_ERR_CUDA;
  p.status = &call->acc;
  p.call = call;
  p.q = q;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.o_part = reinterpret_cast<float *>(parts);
  p.ml_part = reinterpret_cast<float *>(parts + w.o_bytes);
  p.out = out;
  p.lse = lse;
  p.batch = batch;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_ctx_len = max_ctx_len;
  p.num_blocks = num_blocks;
  p.split_tokens = w.split_tokens;
  p.max_splits = w.max_splits;
  p.scale_log2 = scale * kLog2e;
  cudaError_t e = launch_decode(tk, tv, p, d, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free paged decode: the split partial states go to a static
// device array instead of a caller workspace.  For callers that cannot call
// cudaMalloc (a plugin whose host framework owns all device memory, or a
// decode loop that must avoid cudaMalloc/cudaFree and their implicit device
// synchronisation).  Every call on a device shares this one array.
namespace fa {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[FA_DECODE_NOALLOC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device.  In host code the
// symbol is only a host-side stand-in, so the address is looked up once per
// device with cudaGetSymbolAddress while that device is current.
unsigned char *noalloc_scratch() {
  constexpr int kMaxDev = 64;
  static unsigned char *ptrs[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    ptrs[dev] = static_cast<unsigned char *>(p);
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace fa

extern "C" int fa_decode_paged_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                       const int32_t *block_table, int max_blocks_per_seq,
                                       const int32_t *ctx_lens, int max_ctx_len, int batch,
                                       int H, int Hkv, int d, int block_size, int num_blocks,
                                       float scale, void *out, float *lse, fa_stream_t stream) {
  // Same argument rules as fa_decode_paged (checked there); only the size of
  // the partial states must fit the static array.
  if (batch < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || max_ctx_len < 0)
    return FA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || block_size != kDecodeBlock || max_ctx_len > kMaxCtxLen)
    return FA_ERR_UNSUPPORTED;
  if (batch == 0) return FA_OK;
  const DecodeWs w = decode_ws(batch, H, Hkv, d, max_ctx_len);
  const size_t need = FA_WORKSPACE_HEADER_BYTES + w.o_bytes + w.ml_bytes;
  if (need > FA_DECODE_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  unsigned char *scratch = noalloc_scratch();
  if (scratch == nullptr) return FA_ERR_CUDA;
  return fa_decode_paged(q, k_pool, v_pool, block_table, max_blocks_per_seq, ctx_lens,
                         max_ctx_len, batch, H, Hkv, d, block_size, num_blocks, scale, out, lse,
                         scratch, FA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
