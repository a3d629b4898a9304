"""Seeded synthetic inputs and work counters for the attention workloads.

This module only draws random numbers, rounds them to bfloat16 and lays them
out; it holds none of the attention arithmetic.  Both the CUDA path (through
the tests and ``bench.py``) and the CPU oracle (through the tests) take their
inputs from here, so the two sides see identical bf16 bits.

Recipe (all values iid N(0, 1) drawn as float32 and rounded to bf16, round to
nearest even):

* every tensor is generated in chunks of ``CHUNK`` elements; chunk ``c`` of
  stream ``s`` under seed ``seed`` comes from
  ``numpy.random.default_rng(SeedSequence([seed, s, c])).standard_normal``,
  so the bits do not depend on how many threads fill the chunks;
* Q, K, V use seed 0 with streams 0, 1, 2;
* long-context prefill: for each (batch, kv head), ceil(1% of N) key rows
  chosen uniformly without replacement under seed 1 are multiplied by 8
  (exact in bf16), which moves the running row maximum late in many rows;
* varlen: 32 sequence lengths ``rng.integers(64, 4097)`` under seed 2;
* paged decode: context lengths ``rng.integers(512, 32769)`` under seed 3;
  the pool holds exactly sum(ceil(ctx / 16)) blocks and the block table is
  a permutation of the pool under seed 4 (unused table slots hold -1).
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22

# The benchmark/parity workloads, named by what they are.
WORKLOADS = {
    "pr1": dict(kind="dense", B=1, H=1, Hkv=1, N=256, d=64, causal=False),
    "dense_d64": dict(kind="dense", B=4, H=16, Hkv=16, N=2048, d=64, causal=None),
    "long_causal_d128": dict(kind="dense", B=2, H=32, Hkv=32, N=8192, d=128, causal=True,
                             outlier_frac=0.01, outlier_scale=8.0),
    "varlen_gqa_d128": dict(kind="varlen", num_seqs=32, len_lo=64, len_hi=4096, H=16, Hkv=4,
                            d=128, causal=True),
    "paged_decode_gqa_d128": dict(kind="decode", batch=64, H=32, Hkv=8, d=128, block_size=16,
                                  ctx_lo=512, ctx_hi=32768),
    # chunked prefill over a paged cache: each sequence has a cached prefix of
    # U[1024, 16384] tokens (seed 6) and appends a chunk of 1024 new tokens
    "splitkv_small_bh_d128": dict(kind="dense", B=1, H=4, Hkv=4, N=8192, d=128, causal=True),
    "long_causal_fp8_d128": dict(kind="dense_fp8", B=2, H=32, Hkv=32, N=8192, d=128,
                                 causal=True),
    "paged_prefill_gqa_d128": dict(kind="paged_prefill", batch=8, H=32, Hkv=8, d=128,
                                   block_size=16, prefix_lo=1024, prefix_hi=16384, chunk=1024),
}


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def normal_bf16_bits(shape, seed: int, stream: int) -> np.ndarray:
    """N(0,1) samples rounded to bf16, as uint16 bits, chunked and seeded."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16)
    n_chunks = (n + CHUNK - 1) // CHUNK

    def fill(c):
        a = c * CHUNK
        e = min(n, a + CHUNK)
        rng = np.random.default_rng(np.random.SeedSequence([seed, stream, c]))
        out[a:e] = f32_to_bf16_bits(rng.standard_normal(e - a, dtype=np.float32))

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def scale_bf16_bits_pow2(bits: np.ndarray, factor: float) -> np.ndarray:
    """Multiply bf16 values by a power of two (exact, no overflow here)."""
    return f32_to_bf16_bits(bf16_bits_to_f32(bits) * np.float32(factor))


@dataclass
class DenseInputs:
    B: int
    N: int
    H: int
    Hkv: int
    d: int
    q: np.ndarray   # uint16 bf16 bits [B, N, H, d]
    k: np.ndarray   # [B, N, Hkv, d]
    v: np.ndarray   # [B, N, Hkv, d]
    outlier_rows: dict = field(default_factory=dict)


def dense_inputs(B, N, H, Hkv, d, seed=0, outlier_frac=0.0, outlier_scale=8.0,
                 outlier_seed=1) -> DenseInputs:
    q = normal_bf16_bits((B, N, H, d), seed, 0)
    k = normal_bf16_bits((B, N, Hkv, d), seed, 1)
    v = normal_bf16_bits((B, N, Hkv, d), seed, 2)
    rows = {}
    if outlier_frac > 0.0:
        rng = np.random.default_rng(outlier_seed)
        n_out = int(math.ceil(outlier_frac * N))
        for b in range(B):
            for g in range(Hkv):
                idx = np.sort(rng.choice(N, size=n_out, replace=False))
                rows[(b, g)] = idx
                k[b, idx, g, :] = scale_bf16_bits_pow2(k[b, idx, g, :], outlier_scale)
    return DenseInputs(B, N, H, Hkv, d, q, k, v, rows)


# ---------------------------------------------------------------- e4m3 inputs
# OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
# no infinities, codes 0x7f / 0xff are NaN, largest finite 448.
E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """The real value of each of the 256 codes (float64; NaN for 0x7f, 0xff)."""
    c = np.arange(256)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where(c >= 128, -mag, mag)
    val[(c & 0x7f) == 0x7f] = np.nan
    return val


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 code (ties to the even code, the sign kept
    on zero), saturating at +-448.  The input is taken as float32.  Normal
    range (|x| >= 2^-6): the float32 mantissa is rounded to 3 bits (ties to
    even) and the exponent rebiased from 127 to 7; below it the value is a
    multiple of the subnormal step 2^-9."""
    xf = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(xf), np.float32(E4M3_MAX))
    bits = a.view(np.uint32)
    r = (bits + np.uint32(0x7FFFF) + ((bits >> np.uint32(20)) & np.uint32(1))) >> np.uint32(20)
    # r = 8 * biased float32 exponent + 3 mantissa bits; rebias 127 -> 7
    code = np.where(a >= np.float32(2.0 ** -6), r - np.uint32(120 << 3),
                    np.rint(a * np.float32(512.0)).astype(np.uint32)).astype(np.uint8)
    return np.where(np.signbit(xf), code | np.uint8(0x80), code)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return e4m3_values()[np.asarray(codes, dtype=np.int64)]


@dataclass
class Fp8Inputs:
    B: int
    N: int
    H: int
    Hkv: int
    d: int
    q: np.ndarray   # uint8 e4m3 codes [B, N, H, d]
    k: np.ndarray   # [B, N, Hkv, d]
    v: np.ndarray   # [B, N, Hkv, d]
    q_descale: float
    k_descale: float
    v_descale: float
    scale: float | None = None   # softmax scale; None means 1/sqrt(d)

    def real(self, name: str) -> np.ndarray:
        """Dequantised float64 values code * descale of q, k or v."""
        return e4m3_decode(getattr(self, name)) * getattr(self, name + "_descale")


def fp8_inputs(B, N, H, Hkv, d, seed=0) -> Fp8Inputs:
    """N(0, 1) draws (the bf16 recipe's streams 0, 1, 2) quantised per tensor:
    descale = amax / 448 rounded up to a power of two, code = e4m3(x / descale)."""
    out = {}
    for name, shape, stream in (("q", (B, N, H, d), 0), ("k", (B, N, Hkv, d), 1),
                                ("v", (B, N, Hkv, d), 2)):
        x = bf16_bits_to_f32(normal_bf16_bits(shape, seed, stream)).reshape(-1)
        amax = float(np.abs(x).max()) if x.size else 1.0
        ds = 2.0 ** math.ceil(math.log2(max(amax, 1e-30) / E4M3_MAX))
        inv = np.float32(1.0 / ds)    # a power of two: x * inv is exact
        codes = np.empty(x.shape, dtype=np.uint8)
        for c0 in range(0, x.size, CHUNK):
            codes[c0:c0 + CHUNK] = e4m3_encode(x[c0:c0 + CHUNK] * inv)
        out[name] = (codes.reshape(shape), ds)
    return Fp8Inputs(B, N, H, Hkv, d, out["q"][0], out["k"][0], out["v"][0],
                     out["q"][1], out["k"][1], out["v"][1])


def fp8_exact_p_inputs(B, N, H, Hkv, d, seed=0, q_nnz=4) -> Fp8Inputs:
    """Inputs whose softmax weights are powers of two, exact in e4m3: each
    query row has ``q_nnz`` entries of +-1 (descale 1/2), keys are -1, 0, +1
    (descale 2) and the softmax scale is ln 2, so every base-2 score
    q.k * scale * log2(e) is an integer in [-q_nnz, q_nnz].  Values are
    integers in [-8, 8] (exact in e4m3) with descale 1/4."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7]))
    one, m_one = 0x38, 0xB8
    q = np.zeros((B, N, H, d), dtype=np.uint8)
    if B * N * H:
        pos = np.argsort(rng.random((B, N, H, d)), axis=-1)[..., :q_nnz]
        sign = rng.integers(0, 2, size=pos.shape)
        np.put_along_axis(q, pos, np.where(sign == 1, one, m_one).astype(np.uint8), axis=-1)
    kc = rng.integers(-1, 2, size=(B, N, Hkv, d))
    k = np.select([kc == 1, kc == -1], [one, m_one], 0).astype(np.uint8)
    v = e4m3_encode(rng.integers(-8, 9, size=(B, N, Hkv, d)).astype(np.float64))
    return Fp8Inputs(B, N, H, Hkv, d, q, k, v, 0.5, 2.0, 0.25, scale=math.log(2.0))


def varlen_lengths(num_seqs=32, lo=64, hi=4096, seed=2) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=num_seqs).astype(np.int64)


def cu_seqlens_from(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


@dataclass
class VarlenInputs:
    lengths: np.ndarray
    cu_seqlens: np.ndarray
    H: int
    Hkv: int
    d: int
    q: np.ndarray   # [T, H, d]
    k: np.ndarray   # [T, Hkv, d]
    v: np.ndarray

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return int(self.lengths.max()) if len(self.lengths) else 0


def varlen_inputs(lengths, H, Hkv, d, seed=0) -> VarlenInputs:
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = cu_seqlens_from(lengths)
    t = int(cu[-1])
    return VarlenInputs(lengths, cu, H, Hkv, d,
                        normal_bf16_bits((t, H, d), seed, 0),
                        normal_bf16_bits((t, Hkv, d), seed, 1),
                        normal_bf16_bits((t, Hkv, d), seed, 2))


def decode_ctx_lens(batch=64, lo=512, hi=32768, seed=3) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def paged_block_table(ctx_lens, block_size=16, seed=4, max_blocks_per_seq=None):
    """Random-permutation block table; returns (table int32 [batch, max_blocks], num_blocks)."""
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    nblk = (ctx + block_size - 1) // block_size
    num_blocks = int(nblk.sum())
    mb = int(nblk.max()) if len(nblk) else 0
    if max_blocks_per_seq is not None:
        mb = max(mb, int(max_blocks_per_seq))
    perm = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
    table = np.full((len(ctx), max(mb, 1)), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return table, num_blocks


@dataclass
class DecodeInputs:
    batch: int
    H: int
    Hkv: int
    d: int
    block_size: int
    ctx_lens: np.ndarray      # int32 [batch]
    block_table: np.ndarray   # int32 [batch, max_blocks]
    num_blocks: int
    q: np.ndarray             # bf16 bits [batch, H, d]
    k_pool: np.ndarray        # bf16 bits [num_blocks, block_size, Hkv, d]
    v_pool: np.ndarray

    @property
    def max_ctx_len(self) -> int:
        return int(self.ctx_lens.max()) if len(self.ctx_lens) else 0


def decode_inputs(ctx_lens, H, Hkv, d, block_size=16, seed=0, table_seed=4,
                  extra_blocks=0) -> DecodeInputs:
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    table, nb = paged_block_table(ctx, block_size, table_seed)
    nb_total = max(nb + int(extra_blocks), 1)
    return DecodeInputs(len(ctx), H, Hkv, d, block_size, ctx, table, nb_total,
                        normal_bf16_bits((len(ctx), H, d), seed, 0),
                        normal_bf16_bits((nb_total, block_size, Hkv, d), seed, 1),
                        normal_bf16_bits((nb_total, block_size, Hkv, d), seed, 2))


@dataclass
class PagedPrefillInputs:
    pool: DecodeInputs           # pool, block table and ctx_lens (= prefix + chunk)
    q_lens: np.ndarray           # int32 [batch]
    cu_seqlens_q: np.ndarray     # int32 [batch + 1]
    q: np.ndarray                # bf16 bits [total_q, H, d]

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max()) if len(self.q_lens) else 0


def paged_prefill_inputs(ctx_lens, q_lens, H, Hkv, d, block_size=16, seed=0, table_seed=4,
                         extra_blocks=0) -> PagedPrefillInputs:
    """Query chunks over a paged pool: the pool and table follow the decode
    recipe; the packed queries use seed ``seed`` stream 3."""
    pool = decode_inputs(ctx_lens, H, Hkv, d, block_size, seed, table_seed, extra_blocks)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    cu = cu_seqlens_from(q_lens)
    return PagedPrefillInputs(pool, q_lens, cu, normal_bf16_bits((int(cu[-1]), H, d), seed, 3))


def paged_prefill_lengths(batch=8, prefix_lo=1024, prefix_hi=16384, chunk=1024, seed=6):
    prefix = np.random.default_rng(seed).integers(prefix_lo, prefix_hi + 1, size=batch)
    q_lens = np.full(batch, chunk, dtype=np.int32)
    return (prefix + chunk).astype(np.int32), q_lens


# ---------------------------------------------------------------- counters

def prefill_flops(B, N, H, d, causal) -> float:
    """Exact attention work, 4*N^2*d per (batch, head), halved for causal."""
    f = 4.0 * N * N * d * H * B
    return f / 2 if causal else f


def varlen_flops(lengths, H, d, causal) -> float:
    return float(sum(prefill_flops(1, int(L), H, d, causal) for L in lengths))


def paged_prefill_flops(ctx_lens, q_lens, H, d, causal=True) -> float:
    """4*d*H per visible (query, key) pair; bottom-right causal alignment."""
    total = 0.0
    for ctx, nq in zip(ctx_lens, q_lens):
        ctx, nq = int(ctx), int(nq)
        if causal:
            i = np.arange(nq)
            vis = np.clip(i + 1 + (ctx - nq), 0, ctx)
            total += float(vis.sum())
        else:
            total += float(ctx) * nq
    return 4.0 * d * H * total


def decode_bytes(ctx_lens, H, Hkv, d, max_blocks_per_seq, block_size=16) -> int:
    """Algorithmic HBM bytes of one paged decode step.

    K and V rows of every cached token (bf16), the query and output rows
    (bf16), the fp32 LSE, the context lengths and the block-table entries
    that are actually read.
    """
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    kv = int(ctx.sum()) * Hkv * d * 2 * 2
    qo = len(ctx) * H * d * 2 * 2
    lse = len(ctx) * H * 4
    table = int(((ctx + block_size - 1) // block_size).sum()) * 4
    return kv + qo + lse + len(ctx) * 4 + table
