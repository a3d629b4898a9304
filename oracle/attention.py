"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: it is used by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It
shares no code with the CUDA library and imports nothing from it.

What it computes is the plain definition that the FlashAttention pages say
the tiled method reaches exactly (up to floating-point reassociation):

* "S12 FlashAttention" (llminference.xinbetween.com/en/s12/), section
  "Motivation / The problem": S = q k^T, softmax over each row, multiply by V.
* same page, "Core idea" and the box on FLOPs: the streaming version does the
  same arithmetic as the textbook one and reaches the same result; the
  "What this unlocks" figures say the two differ only in the order in which
  floating-point sums are formed.

So the oracle materialises the whole score matrix for one (sequence, head)
pair at a time, in float64, and applies the textbook softmax.  It never runs
the online recurrence (that lives only in the kernels and, for cross-checking
the oracle, in the tests).

Readings taken where the pages leave a detail open (each is listed again in
the design notes):

* scale: an explicit argument, default 1/sqrt(d) ("Core idea" listing divides
  q k^T by sqrt(d)); the worked example on the explainer page uses scale 1.
* the maximum is taken per query row over *scaled* scores.
* GQA: query head h reads key/value head floor(h / (H / Hkv)).  The section
  "How this composes with what you already built" has a group of query heads
  share one KV head without fixing which; contiguous groups are the plainest
  reading.
* causal masking is bottom-right aligned: key j is visible to query i iff
  j <= i + (Nk - Nq).  For Nq == Nk this is the usual j <= i.
* LSE is the natural-log logsumexp of the scaled scores, M + ln(sum exp(S - M)).
* a query row that sees no key at all gets O = 0 and LSE = -inf (the pages
  only warn that exp(-inf - -inf) is NaN; the oracle never produces NaN).
* paged KV cache: logical token t of sequence b lives in
  pool[block_table[b, t // block_size], t % block_size]; slots of the last
  block past the context length are ignored ("Implementation", the paged
  listing takes n = min(block_size, seq_len - logical * block_size) rows).

Parity status: every public function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (worked example, closed forms, invariants,
brute force, and an independent re-derivation of the pages' recurrence).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attention_one",
    "attention_dense",
    "attention_varlen",
    "paged_decode",
    "paged_prefill",
    "tile_state",
    "merge_states",
    "gather_paged",
]


def _as64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def attention_one(q, k, v, scale=None, causal=False, rows=None, heads=None):
    """Exact attention of one sequence, all heads.

    q: [Nq, H, d]; k, v: [Nk, Hkv, d] (any float dtype, computed in float64).
    Returns (o [Nq, H, d] float64, lse [H, Nq] float64).  ``rows`` / ``heads``
    restrict the work to those query rows / heads (others stay 0 / -inf);
    each selected row keeps its own causal visibility.

    Definition ("S12 FlashAttention", Motivation): S = scale * q k^T,
    P = softmax(S) row-wise, O = P V.  LSE_i = M_i + ln sum_j exp(S_ij - M_i).
    """
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    nq, h_q, d = q.shape
    nk, h_kv, d_k = k.shape
    if d_k != d or v.shape[:2] != (nk, h_kv):
        raise ValueError("shape mismatch between q, k, v")
    if h_q % h_kv != 0:
        raise ValueError("H must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = h_q // h_kv
    dv = v.shape[2]

    o = np.zeros((nq, h_q, dv), dtype=np.float64)
    lse = np.full((h_q, nq), -np.inf, dtype=np.float64)
    if nq == 0:
        return o, lse

    sel = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)
    if causal:
        cols = np.arange(nk)[None, :]
        visible = cols <= sel[:, None] + (nk - nq)
    else:
        visible = np.ones((sel.shape[0], nk), dtype=bool)

    for h in (range(h_q) if heads is None else heads):
        g = h // group
        s = scale * (q[sel, h, :] @ k[:, g, :].T)           # [rows, Nk]
        s = np.where(visible, s, -np.inf)
        row_max = s.max(axis=1) if nk > 0 else np.full(sel.shape[0], -np.inf)
        live = np.isfinite(row_max)
        safe_max = np.where(live, row_max, 0.0)
        e = np.exp(s - safe_max[:, None])                   # masked -> 0
        z = e.sum(axis=1)
        p = np.divide(e, z[:, None], out=np.zeros_like(e), where=live[:, None])
        o[sel, h, :] = p @ v[:, g, :]
        lse[h, sel] = np.where(live, safe_max + np.log(np.where(live, z, 1.0)), -np.inf)
    return o, lse


def attention_dense(q, k, v, scale=None, causal=False):
    """Batched dense layout: q, out [B, N, H, d]; k, v [B, N, Hkv, d].

    Returns (o [B, N, H, d], lse [B, H, N]).  Each batch element is an
    independent sequence evaluated with :func:`attention_one`.
    """
    q = np.asarray(q)
    b_sz = q.shape[0]
    outs, lses = [], []
    for b in range(b_sz):
        o, lse = attention_one(q[b], k[b], v[b], scale=scale, causal=causal)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)


def attention_varlen(q, k, v, cu_seqlens, scale=None, causal=False):
    """Packed variable-length batch (the explainer article's "Varlen" section).

    q: [T, H, d]; k, v: [T, Hkv, d]; cu_seqlens: [S + 1] token offsets.
    Sequence s owns rows [cu[s], cu[s+1]) of q, k and v and attends only to
    its own keys (no cross-sequence attention; causal rule per sequence).
    Returns (o [T, H, d], lse [H, T]).
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    t_total, h_q, _ = q.shape
    o = np.zeros((t_total, h_q, v.shape[2]), dtype=np.float64)
    lse = np.full((h_q, t_total), -np.inf, dtype=np.float64)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        if e <= a:
            continue
        o_s, lse_s = attention_one(q[a:e], k[a:e], v[a:e], scale=scale, causal=causal)
        o[a:e] = o_s
        lse[:, a:e] = lse_s
    return o, lse


def gather_paged(pool, block_table_row, ctx_len, block_size):
    """Contiguous [ctx_len, Hkv, d] view of one sequence of a paged pool.

    Logical token t is pool[block_table_row[t // block_size], t % block_size]
    ("S12 FlashAttention", Implementation: the block table sits in front of
    the key access; the last block contributes only its first n rows).
    """
    pool = np.asarray(pool)
    rows = []
    n_blocks = (int(ctx_len) + block_size - 1) // block_size
    for logical in range(n_blocks):
        physical = int(block_table_row[logical])
        n = min(block_size, int(ctx_len) - logical * block_size)
        rows.append(pool[physical, :n])
    if not rows:
        return np.zeros((0,) + pool.shape[2:], dtype=pool.dtype)
    return np.concatenate(rows, axis=0)


def paged_decode(q, k_pool, v_pool, block_table, ctx_lens, block_size, scale=None,
                 batches=None, heads=None):
    """One query token per sequence against a paged KV cache.

    q: [batch, H, d]; k_pool, v_pool: [num_blocks, block_size, Hkv, d];
    block_table: [batch, max_blocks]; ctx_lens: [batch].
    Every cached key is visible to the single query (decode step).
    Returns (o [batch, H, d], lse [batch, H]); rows not listed in
    ``batches`` / heads not in ``heads`` are left 0 / -inf (for sampling).
    """
    q = np.asarray(q)
    b_sz, h_q, d = q.shape
    o = np.zeros((b_sz, h_q, np.asarray(v_pool).shape[3]), dtype=np.float64)
    lse = np.full((b_sz, h_q), -np.inf, dtype=np.float64)
    sel_b = range(b_sz) if batches is None else batches
    for b in sel_b:
        kc = gather_paged(k_pool, block_table[b], ctx_lens[b], block_size)
        vc = gather_paged(v_pool, block_table[b], ctx_lens[b], block_size)
        o_b, lse_b = attention_one(q[b][None], kc, vc, scale=scale, causal=False)
        if heads is None:
            o[b] = o_b[0]
            lse[b] = lse_b[:, 0]
        else:
            for h in heads:
                o[b, h] = o_b[0, h]
                lse[b, h] = lse_b[h, 0]
    return o, lse


def paged_prefill(q, k_pool, v_pool, block_table, ctx_lens, cu_seqlens_q, block_size,
                  scale=None, causal=True, seqs=None, heads=None):
    """Several query tokens per sequence against a paged KV cache (chunked
    prefill over cached keys).

    "S12 FlashAttention", Implementation: the paged variant is the same loop
    with the block table in front of the key access; here each sequence b
    brings ``cu_seqlens_q[b+1] - cu_seqlens_q[b]`` query tokens (packed like
    the varlen layout) and reads its ``ctx_lens[b]`` cached keys through the
    block table.  Causal masking is bottom-right aligned: query i of a chunk
    of Nq queries sees key j iff j <= i + (ctx - Nq), so the chunk's queries
    are the last Nq positions of the sequence.
    q: [Tq, H, d]; pools [num_blocks, block_size, Hkv, d]; returns
    (o [Tq, H, d], lse [H, Tq]).
    """
    q = np.asarray(q)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    t_q, h_q, _ = q.shape
    o = np.zeros((t_q, h_q, np.asarray(v_pool).shape[3]), dtype=np.float64)
    lse = np.full((h_q, t_q), -np.inf, dtype=np.float64)
    for b in (range(len(cu) - 1) if seqs is None else seqs):
        a, e = int(cu[b]), int(cu[b + 1])
        if e <= a:
            continue
        kc = gather_paged(k_pool, block_table[b], ctx_lens[b], block_size)
        vc = gather_paged(v_pool, block_table[b], ctx_lens[b], block_size)
        o_b, lse_b = attention_one(q[a:e], kc, vc, scale=scale, causal=causal, heads=heads)
        o[a:e] = o_b
        lse[:, a:e] = lse_b
    return o, lse


def tile_state(scores, values=None):
    """(m, l, o) of one tile of scores for one query row.

    m = max_j s_j, l = sum_j exp(s_j - m), o = sum_j exp(s_j - m) v_j
    ("S12 FlashAttention" diagram: the running max, running sum and the
    un-normalised weighted sum of v).  An empty or fully masked tile is the
    neutral state (m = -inf, l = 0, o = 0).
    """
    s = _as64(scores).reshape(-1)
    vals = np.zeros((s.shape[0], 0)) if values is None else _as64(values)
    if vals.ndim == 1:
        vals = vals.reshape(-1, 1)
    if s.size == 0 or not np.isfinite(s.max()):
        return -np.inf, 0.0, np.zeros(vals.shape[1])
    m = float(s.max())
    w = np.exp(s - m)
    return m, float(w.sum()), w @ vals


def merge_states(states):
    """Combine partial (m, l, o) states into one.

    Explainer page ("Show the maths"): m_new = max(m, m~),
    l_new = e^(m - m_new) l + e^(m~ - m_new) l~; the same rescaling applies to
    o ("S12 FlashAttention", flash-decoding bullet and exercise 1).  Neutral
    states (m = -inf) contribute nothing.
    """
    states = list(states)
    if not states:
        raise ValueError("no states")
    m_all = max(float(m) for m, _, _ in states)
    dim = np.asarray(states[0][2]).shape
    if not np.isfinite(m_all):
        return -np.inf, 0.0, np.zeros(dim)
    l_tot = 0.0
    o_tot = np.zeros(dim)
    for m, l, o in states:
        if not np.isfinite(m):
            continue
        w = math.exp(float(m) - m_all)
        l_tot += w * float(l)
        o_tot = o_tot + w * _as64(o)
    return m_all, l_tot, o_tot
