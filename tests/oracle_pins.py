"""Pins for the fp64 oracle: checks that do not trust the oracle itself.

Each ``pin_*`` function takes an oracle namespace (normally the ``oracle``
package) and raises AssertionError when the oracle disagrees with something
the pages or plain mathematics fix.  They are written as functions of the
namespace so that ``test_oracle_mutants.py`` can run them against copies of
the oracle with a planted mistake and show that each mistake is caught.

Sources pinned against:
* the worked example of the FlashAttention explainer page
  (tachyon.techntrek.in/learn/flash-attention, "Show the maths");
* closed forms and invariants of softmax attention;
* per-element brute force in pure Python on tiny inputs;
* an independent fp64 re-derivation of the online recurrence of
  "S12 FlashAttention" (sections "Core idea" and "Implementation"), its
  flash-decoding split ("What this unlocks", exercise 1) and the NaN guard
  ("exp(-inf - -inf) is NaN" box, exercise 2).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- helpers

def rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def brute_attention(q, k, v, scale, causal):
    """Pure-Python per-element attention for one sequence (tiny sizes).

    q [Nq][H][d], k/v [Nk][Hkv][d] as nested lists or arrays.
    """
    nq, h_q, d = len(q), len(q[0]), len(q[0][0])
    nk, h_kv = len(k), len(k[0])
    dv = len(v[0][0])
    group = h_q // h_kv
    o = [[[0.0] * dv for _ in range(h_q)] for _ in range(nq)]
    lse = [[-math.inf] * nq for _ in range(h_q)]
    for h in range(h_q):
        g = h // group
        for i in range(nq):
            scores = []
            for j in range(nk):
                if causal and j > i + (nk - nq):
                    continue
                dot = 0.0
                for c in range(d):
                    dot += float(q[i][h][c]) * float(k[j][g][c])
                scores.append((j, scale * dot))
            if not scores:
                continue
            mx = max(s for _, s in scores)
            z = sum(math.exp(s - mx) for _, s in scores)
            for j, s in scores:
                w = math.exp(s - mx) / z
                for c in range(dv):
                    o[i][h][c] += w * float(v[j][g][c])
            lse[h][i] = mx + math.log(z)
    return np.array(o), np.array(lse)


def recurrence_one_head(q, k, v, scale, tile, causal, guard=True, visible=None):
    """The pages' streaming recurrence, vectorised over query rows.

    q [Nq, d], k/v [Nk, d].  Running max m, running sum l, un-normalised
    accumulator o; alpha = exp(m_old - m_new) rescales everything so far.
    With ``guard`` the reference maximum of a row that has seen only masked
    keys is 0 instead of -inf, so alpha and p stay finite.
    """
    nq, nk = q.shape[0], k.shape[0]
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    o = np.zeros((nq, v.shape[1]))
    rows = np.arange(nq)[:, None]
    for start in range(0, nk, tile):
        stop = min(nk, start + tile)
        s = scale * (q @ k[start:stop].T)
        cols = np.arange(start, stop)[None, :]
        if causal:
            s = np.where(cols <= rows + (nk - nq), s, -np.inf)
        if visible is not None:
            s = np.where(visible[:, start:stop], s, -np.inf)
        with np.errstate(invalid="ignore"):
            m_new = np.maximum(m, s.max(axis=1))
            ref = np.where(np.isfinite(m_new), m_new, 0.0) if guard else m_new
            alpha = np.exp(m - ref)
            p = np.exp(s - ref[:, None])
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ v[start:stop]
        m = m_new
    with np.errstate(invalid="ignore", divide="ignore"):
        out = o / l[:, None]
        lse = np.where(l > 0, m + np.log(l), -np.inf)
    return out, lse


# --------------------------------------------------------------- pins

def pin_worked_example(ora):
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    s = np.array(g["scores"])
    cut = g["tile_boundary"]
    tol = 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12
    pr = g["printed"]
    m1, l1, _ = ora.tile_state(s[:cut])
    m2, l2, _ = ora.tile_state(s[cut:])
    assert abs(m1 - pr["tile1_m"]) <= tol and abs(l1 - pr["tile1_l"]) <= tol, (m1, l1)
    assert abs(m2 - pr["tile2_m"]) <= tol and abs(l2 - pr["tile2_l"]) <= tol, (m2, l2)
    m, l, _ = ora.merge_states([(m1, l1, np.zeros(1)), (m2, l2, np.zeros(1))])
    assert m == max(pr["tile1_m"], pr["tile2_m"])
    assert abs(l - pr["merged_l"]) <= tol, l
    # the merged sum is the full-row sum (same page): one tile over all scores
    mf, lf, _ = ora.tile_state(s)
    assert mf == m and abs(lf - l) <= 1e-12
    # The same row through the attention definition: d = 1, q = 1, k_j = s_j.
    q = np.ones((1, 1, 1))
    k = s.reshape(-1, 1, 1)
    v = np.arange(len(s), dtype=np.float64).reshape(-1, 1, 1)
    o, lse = ora.attention_one(q, k, v, scale=g["scale"], causal=False)
    lse_printed = pr["tile2_m"] + math.log(pr["merged_l"])
    assert abs(lse[0, 0] - lse_printed) <= tol / pr["merged_l"] + 1e-9, lse
    # output = softmax-weighted mean of v_j = j, with weights exp(s_j - 3)/2.611...
    w = np.exp(s - 3.0) / pr["merged_l"]
    assert abs(o[0, 0, 0] - float(w @ np.arange(len(s)))) <= 5e-3


def pin_zero_query(ora):
    """q = 0: every visible key gets the same weight."""
    rng = np.random.default_rng(11)
    nq, nk, h, hkv, d = 5, 7, 4, 2, 3
    q = np.zeros((nq, h, d))
    k = rand(rng, nk, hkv, d)
    v = rand(rng, nk, hkv, d)
    for causal in (False, True):
        o, lse = ora.attention_one(q, k, v, scale=0.7, causal=causal)
        for i in range(nq):
            nvis = (i + (nk - nq) + 1) if causal else nk
            for hh in range(h):
                g = hh // (h // hkv)
                np.testing.assert_allclose(o[i, hh], v[:nvis, g].mean(axis=0), atol=1e-13)
                assert abs(lse[hh, i] - math.log(nvis)) < 1e-13


def pin_single_key(ora):
    rng = np.random.default_rng(12)
    q = rand(rng, 1, 2, 4)
    k = rand(rng, 1, 2, 4)
    v = rand(rng, 1, 2, 4)
    for causal in (False, True):
        o, lse = ora.attention_one(q, k, v, scale=0.5, causal=causal)
        np.testing.assert_allclose(o[0], v[0], atol=1e-15)
        for hh in range(2):
            assert abs(lse[hh, 0] - 0.5 * float(q[0, hh] @ k[0, hh])) < 1e-13


def pin_dominant_key(ora):
    """A key whose score beats all others by > 50 takes all the weight."""
    rng = np.random.default_rng(13)
    nk, d = 9, 4
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.0
    k = rand(rng, nk, 1, d) * 0.1
    k[6, 0, 0] = 80.0
    v = rand(rng, nk, 1, d)
    o, lse = ora.attention_one(q, k, v, scale=1.0)
    np.testing.assert_allclose(o[0, 0], v[6, 0], atol=1e-15)
    assert abs(lse[0, 0] - 80.0) < 1e-12


def pin_constant_values(ora):
    rng = np.random.default_rng(14)
    q = rand(rng, 6, 2, 5)
    k = rand(rng, 6, 1, 5)
    v = np.full((6, 1, 5), 3.25)
    o, _ = ora.attention_one(q, k, v, causal=True)
    np.testing.assert_allclose(o, 3.25, atol=1e-14)


def pin_rows_are_softmax(ora):
    """With V = identity the output is the probability matrix itself."""
    rng = np.random.default_rng(15)
    nq = nk = 6
    q = rand(rng, nq, 1, 3)
    k = rand(rng, nk, 1, 3)
    v = np.eye(nk).reshape(nk, 1, nk)
    for causal in (False, True):
        p, lse = ora.attention_one(q, k, v, scale=1.3, causal=causal)
        p = p[:, 0, :]
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
        if causal:
            assert np.all(np.triu(p, 1) == 0)
        # ratios of probabilities follow the score differences exactly
        s = 1.3 * (q[:, 0] @ k[:, 0].T)
        for i in range(nq):
            j_max = i + 1 if causal else nk
            np.testing.assert_allclose(np.log(p[i, :j_max]) - np.log(p[i, 0]),
                                       s[i, :j_max] - s[i, 0], atol=1e-11)
            assert abs(lse[0, i] - (s[i, 0] - math.log(p[i, 0]))) < 1e-11


def pin_convex_combination(ora):
    rng = np.random.default_rng(16)
    q = rand(rng, 20, 3, 8)
    k = rand(rng, 20, 3, 8)
    v = rand(rng, 20, 3, 8)
    o, _ = ora.attention_one(q, k, v, causal=True)
    for i in range(20):
        lo = v[:i + 1].min(axis=0)
        hi = v[:i + 1].max(axis=0)
        assert np.all(o[i] >= lo - 1e-12) and np.all(o[i] <= hi + 1e-12)


def pin_key_permutation(ora):
    rng = np.random.default_rng(17)
    q = rand(rng, 4, 2, 6)
    k = rand(rng, 11, 2, 6)
    v = rand(rng, 11, 2, 6)
    perm = rng.permutation(11)
    o1, l1 = ora.attention_one(q, k, v)
    o2, l2 = ora.attention_one(q, k[perm], v[perm])
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def pin_masked_keys_do_nothing(ora):
    """Causal: changing keys/values a row cannot see leaves that row alone.
    Varlen: another sequence's tokens never reach this one."""
    rng = np.random.default_rng(18)
    q = rand(rng, 10, 2, 4)
    k = rand(rng, 10, 2, 4)
    v = rand(rng, 10, 2, 4)
    o1, l1 = ora.attention_one(q, k, v, causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[6:] = 1e3
    v2[6:] = -7.0
    o2, l2 = ora.attention_one(q, k2, v2, causal=True)
    np.testing.assert_array_equal(o1[:6], o2[:6])
    np.testing.assert_array_equal(l1[:, :6], l2[:, :6])
    assert not np.allclose(o1[6:], o2[6:])
    lengths = [3, 5, 4]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    qv = rand(rng, cu[-1], 2, 4)
    kv = rand(rng, cu[-1], 1, 4)
    vv = rand(rng, cu[-1], 1, 4)
    for causal in (False, True):
        ov, lv = ora.attention_varlen(qv, kv, vv, cu, scale=0.4, causal=causal)
        for s in range(len(lengths)):
            a, e = cu[s], cu[s + 1]
            o_s, l_s = ora.attention_one(qv[a:e], kv[a:e], vv[a:e], scale=0.4, causal=causal)
            np.testing.assert_array_equal(ov[a:e], o_s)
            np.testing.assert_array_equal(lv[:, a:e], l_s)


def pin_brute_force(ora):
    rng = np.random.default_rng(19)
    cases = [(1, 1, 1, 1, 1), (4, 4, 2, 1, 3), (3, 7, 4, 2, 4), (8, 8, 2, 2, 2), (5, 2, 3, 3, 4)]
    for (nq, nk, h, hkv, d) in cases:
        q = rand(rng, nq, h, d)
        k = rand(rng, nk, hkv, d)
        v = rand(rng, nk, hkv, d + 1)
        for causal in (False, True):
            o_ref, l_ref = brute_attention(q, k, v, 0.9, causal)
            o, l = ora.attention_one(q, k, v, scale=0.9, causal=causal)
            np.testing.assert_allclose(o, o_ref, atol=1e-13, rtol=0)
            np.testing.assert_allclose(l, l_ref, atol=1e-13, rtol=0)


def pin_default_scale(ora):
    rng = np.random.default_rng(20)
    q = rand(rng, 3, 1, 16)
    k = rand(rng, 5, 1, 16)
    v = rand(rng, 5, 1, 16)
    o, l = ora.attention_one(q, k, v)
    o_ref, l_ref = brute_attention(q, k, v, 0.25, False)
    np.testing.assert_allclose(o, o_ref, atol=1e-13)
    np.testing.assert_allclose(l, l_ref, atol=1e-13)


def pin_recurrence(ora):
    """Naive (oracle) == the pages' tiled recurrence at every tile size."""
    rng = np.random.default_rng(21)
    for (nq, nk, h, hkv, d) in [(37, 37, 4, 2, 16), (64, 64, 2, 1, 32), (20, 45, 2, 2, 8)]:
        q = rand(rng, nq, h, d, scale=2.0)
        k = rand(rng, nk, hkv, d, scale=2.0)
        v = rand(rng, nk, hkv, d)
        for causal in (False, True):
            o, l = ora.attention_one(q, k, v, scale=0.3, causal=causal)
            for tile in (1, 3, 16, 64):
                for hh in range(h):
                    g = hh // (h // hkv)
                    o_t, l_t = recurrence_one_head(q[:, hh], k[:, g], v[:, g], 0.3, tile, causal)
                    np.testing.assert_allclose(o_t, o[:, hh], atol=1e-12, rtol=0)
                    np.testing.assert_allclose(l_t, l[hh], atol=1e-12, rtol=0)


def pin_paged(ora):
    """Paged decode == the pages' paged recurrence over the block table, and
    slots of the last block past the context length are never used."""
    rng = np.random.default_rng(22)
    bs, hkv, h, d = 4, 2, 4, 8
    ctx = np.array([1, 4, 5, 11, 16])
    nblk = (ctx + bs - 1) // bs
    nb = int(nblk.sum()) + 3
    perm = rng.permutation(nb)
    table = np.full((len(ctx), int(nblk.max())), -1)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    kp = rand(rng, nb, bs, hkv, d)
    vp = rand(rng, nb, bs, hkv, d)
    q = rand(rng, len(ctx), h, d)
    o, l = ora.paged_decode(q, kp, vp, table, ctx, bs, scale=0.5)
    # poison every slot past the context length: nothing may change
    kp2, vp2 = kp.copy(), vp.copy()
    for b, c in enumerate(ctx):
        last = table[b, (c - 1) // bs]
        kp2[last, c - ((c - 1) // bs) * bs:] = np.nan
        vp2[last, c - ((c - 1) // bs) * bs:] = np.nan
    unused = sorted(set(range(nb)) - set(table[table >= 0].tolist()))
    kp2[unused] = np.nan
    vp2[unused] = np.nan
    o2, l2 = ora.paged_decode(q, kp2, vp2, table, ctx, bs, scale=0.5)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)
    for b, c in enumerate(ctx):
        for hh in range(h):
            g = hh // (h // hkv)
            m_r, l_r = -np.inf, 0.0
            o_r = np.zeros(d)
            for logical, physical in enumerate(table[b]):
                n = min(bs, c - logical * bs)
                if n <= 0:
                    break
                s = 0.5 * (kp[physical, :n, g] @ q[b, hh])
                m_new = max(m_r, s.max())
                alpha = math.exp(m_r - m_new) if np.isfinite(m_r) else 0.0
                p = np.exp(s - m_new)
                l_r, o_r, m_r = alpha * l_r + p.sum(), alpha * o_r + p @ vp[physical, :n, g], m_new
            np.testing.assert_allclose(o[b, hh], o_r / l_r, atol=1e-12, rtol=0)
            assert abs(l[b, hh] - (m_r + math.log(l_r))) < 1e-12


def pin_flash_decoding(ora):
    """Split the keys over four workers, merge their (m, l, o): same answer."""
    rng = np.random.default_rng(23)
    nk, d = 103, 8
    q = rand(rng, 1, 1, d, scale=3.0)
    k = rand(rng, nk, 1, d)
    v = rand(rng, nk, 1, d)
    o, lse = ora.attention_one(q, k, v, scale=0.5)
    s = 0.5 * (k[:, 0] @ q[0, 0])
    bounds = [0, 7, 50, 51, nk]
    states = [ora.tile_state(s[a:e], v[a:e, 0]) for a, e in zip(bounds[:-1], bounds[1:])]
    states.append(ora.tile_state(s[:0], v[:0, 0]))          # an empty split
    m, l, acc = ora.merge_states(states)
    np.testing.assert_allclose(acc / l, o[0, 0], atol=1e-13)
    assert abs(m + math.log(l) - lse[0, 0]) < 1e-13
    # merging is order independent and associative
    m2, l2, acc2 = ora.merge_states([ora.merge_states(states[2:]), ora.merge_states(states[:2])])
    assert m2 == m and abs(l2 - l) < 1e-12
    np.testing.assert_allclose(acc2, acc, atol=1e-12)


def pin_nan_guard(ora):
    """A fully masked first tile: NaN without the guard, the oracle's answer with it."""
    rng = np.random.default_rng(24)
    nk, d = 12, 4
    q = rand(rng, 1, d)
    k = rand(rng, nk, d)
    v = rand(rng, nk, d)
    visible = np.zeros((1, nk), dtype=bool)
    visible[0, 4:] = True                                   # first tile of 4 all masked
    o_bad, _ = recurrence_one_head(q, k, v, 1.0, 4, False, guard=False, visible=visible)
    assert np.isnan(o_bad).all()
    o_ok, l_ok = recurrence_one_head(q, k, v, 1.0, 4, False, guard=True, visible=visible)
    o_ref, l_ref = ora.attention_one(q[:, None], k[4:, None], v[4:, None], scale=1.0)
    np.testing.assert_allclose(o_ok, o_ref[:, 0], atol=1e-13)
    np.testing.assert_allclose(l_ok, l_ref[0], atol=1e-13)


def pin_fully_masked_row(ora):
    """More queries than keys with bottom-right causal alignment: the first
    rows see nothing and must come out as O = 0, LSE = -inf (never NaN)."""
    rng = np.random.default_rng(25)
    q = rand(rng, 5, 1, 3)
    k = rand(rng, 2, 1, 3)
    v = rand(rng, 2, 1, 3)
    o, l = ora.attention_one(q, k, v, causal=True)
    assert np.all(o[:3] == 0) and np.all(np.isneginf(l[0, :3]))
    assert np.all(np.isfinite(o[3:])) and np.all(np.isfinite(l[0, 3:]))
    np.testing.assert_allclose(o[3, 0], v[0, 0], atol=1e-15)


def pin_dense_layout(ora):
    rng = np.random.default_rng(26)
    q = rand(rng, 2, 6, 4, 3)
    k = rand(rng, 2, 6, 2, 3)
    v = rand(rng, 2, 6, 2, 3)
    o, l = ora.attention_dense(q, k, v, causal=True)
    assert o.shape == (2, 6, 4, 3) and l.shape == (2, 4, 6)
    for b in range(2):
        o_ref, l_ref = brute_attention(q[b], k[b], v[b], 1 / math.sqrt(3), True)
        np.testing.assert_allclose(o[b], o_ref, atol=1e-13)
        np.testing.assert_allclose(l[b], l_ref, atol=1e-13)


def pin_paged_prefill(ora):
    """Chunked prefill over a paged cache: (1) a chunk covering the whole
    sequence laid out contiguously is plain causal attention; (2) per element
    it matches a pure-Python evaluation of the bottom-right causal rule;
    (3) a decode step (chunk of one query) matches paged_decode; (4) stale
    slots past the context never matter."""
    rng = np.random.default_rng(27)
    bs, hkv, h, d = 4, 2, 4, 3
    ctx = np.array([9, 4, 13])
    qlen = np.array([3, 4, 1])
    nblk = (ctx + bs - 1) // bs
    nb = int(nblk.sum()) + 2
    perm = rng.permutation(nb)
    table = np.full((3, int(nblk.max())), -1)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    kp = rand(rng, nb, bs, hkv, d)
    vp = rand(rng, nb, bs, hkv, d)
    cu = np.concatenate([[0], np.cumsum(qlen)])
    q = rand(rng, int(cu[-1]), h, d)
    o, l = ora.paged_prefill(q, kp, vp, table, ctx, cu, bs, scale=0.7, causal=True)
    for b in range(3):
        kc = np.concatenate([kp[table[b, t // bs], t % bs][None] for t in range(ctx[b])])
        vc = np.concatenate([vp[table[b, t // bs], t % bs][None] for t in range(ctx[b])])
        o_ref, l_ref = brute_attention(q[cu[b]:cu[b + 1]], kc, vc, 0.7, True)
        np.testing.assert_allclose(o[cu[b]:cu[b + 1]], o_ref, atol=1e-13)
        np.testing.assert_allclose(l[:, cu[b]:cu[b + 1]], l_ref, atol=1e-13)
    # one query per sequence is a decode step
    od, ld = ora.paged_decode(q[cu[1:] - 1], kp, vp, table, ctx, bs, scale=0.7)
    np.testing.assert_allclose(o[cu[1:] - 1], od, atol=1e-13)
    np.testing.assert_allclose(l[:, cu[1:] - 1].T, ld, atol=1e-13)
    # whole sequence as the chunk over a contiguous pool == causal attention
    kfull = rand(rng, 8, 1, 2)
    vfull = rand(rng, 8, 1, 2)
    qfull = rand(rng, 8, 2, 2)
    o1, l1 = ora.paged_prefill(qfull, kfull.reshape(2, 4, 1, 2), vfull.reshape(2, 4, 1, 2),
                               np.array([[0, 1]]), np.array([8]), np.array([0, 8]), 4)
    o2, l2 = ora.attention_one(qfull, kfull, vfull, causal=True)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


ALL_PINS = [
    pin_worked_example, pin_zero_query, pin_single_key, pin_dominant_key,
    pin_constant_values, pin_rows_are_softmax, pin_convex_combination,
    pin_key_permutation, pin_masked_keys_do_nothing, pin_brute_force,
    pin_default_scale, pin_recurrence, pin_paged, pin_flash_decoding,
    pin_nan_guard, pin_fully_masked_row, pin_dense_layout, pin_paged_prefill,
]


# ------------------------------------------------------------ backward pass
# Pins for ``oracle.attention_grad``.  Each takes the forward oracle (for
# attention_one) and the gradient oracle (for attention_backward_one); the
# finite differences use only the forward definition.

def _loss(fwd, q, k, v, do, scale, causal):
    o, _ = fwd.attention_one(q, k, v, scale=scale, causal=causal)
    return float((o * do).sum())


def pin_backward_finite_differences(fwd, bwd):
    """Central differences of <O, dO> w.r.t. every input element agree with
    the analytic gradient (GQA, causal with Nq < Nk, and non-causal)."""
    rng = np.random.default_rng(41)
    eps = 1e-6
    for nq, nk, h, hkv, causal in ((5, 5, 2, 1, True), (3, 6, 2, 2, True), (4, 4, 3, 1, False)):
        q, k, v = rand(rng, nq, h, 3), rand(rng, nk, hkv, 3), rand(rng, nk, hkv, 3)
        do = rand(rng, nq, h, 3)
        scale = 0.7
        dq, dk, dv = bwd.attention_backward_one(q, k, v, do, scale=scale, causal=causal)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args = {"q": q, "k": k, "v": v}
                args[name] = xp
                lp = _loss(fwd, args["q"], args["k"], args["v"], do, scale, causal)
                args[name] = xm
                lm = _loss(fwd, args["q"], args["k"], args["v"], do, scale, causal)
                num[idx] = (lp - lm) / (2 * eps)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=f"d{name}")


def pin_backward_invariants(fwd, bwd):
    """Rows of P sum to 1, so the value gradients of a KV head add up to the
    upstream gradients of its query heads; without a mask, moving every key
    by one vector leaves the softmax unchanged, so the key gradients sum to
    zero.  The gradient is linear in dO."""
    rng = np.random.default_rng(43)
    q, k, v = rand(rng, 7, 4, 5), rand(rng, 9, 2, 5), rand(rng, 9, 2, 5)
    do = rand(rng, 7, 4, 5)
    for causal in (False, True):
        dq, dk, dv = bwd.attention_backward_one(q, k, v, do, causal=causal)
        for g in range(2):
            np.testing.assert_allclose(dv[:, g].sum(axis=0), do[:, 2 * g:2 * g + 2].sum(axis=(0, 1)),
                                       atol=1e-12)
        if not causal:
            np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
        dq2, dk2, dv2 = bwd.attention_backward_one(q, k, v, 3.0 * do, causal=causal)
        np.testing.assert_allclose(dq2, 3.0 * dq, atol=1e-12)
        np.testing.assert_allclose(dk2, 3.0 * dk, atol=1e-12)
    # a single visible key: O = v_0, so dV_0 = dO and dQ = dK = 0
    dq, dk, dv = bwd.attention_backward_one(q[:1], k[:1], v[:1], do[:1], causal=True)
    np.testing.assert_allclose(dv[0], do[0].reshape(2, 2, 5).sum(axis=1), atol=1e-12)
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)
    np.testing.assert_allclose(dk, 0.0, atol=1e-12)


def pin_backward_dense_layout(fwd, bwd):
    rng = np.random.default_rng(47)
    q, k, v, do = rand(rng, 2, 6, 2, 3), rand(rng, 2, 6, 1, 3), rand(rng, 2, 6, 1, 3), rand(rng, 2, 6, 2, 3)
    dq, dk, dv = bwd.attention_backward_dense(q, k, v, do, causal=True)
    for b in range(2):
        r = bwd.attention_backward_one(q[b], k[b], v[b], do[b], causal=True)
        for x, y in zip((dq[b], dk[b], dv[b]), r):
            np.testing.assert_allclose(x, y, atol=0)


def pin_backward_varlen_finite_differences(fwd, bwd):
    """The packed gradient against central differences of <O, dO> through the
    packed forward oracle (sequences of 3, 0, 1 and 4 rows, GQA, both masks):
    a row slice taken from the wrong sequence, or a key seen across a
    sequence boundary, moves the loss where the analytic gradient says it
    does not."""
    rng = np.random.default_rng(53)
    cu = np.array([0, 3, 3, 4, 8])
    t = int(cu[-1])
    eps = 1e-6
    scale = 0.8
    for causal in (False, True):
        q, k, v = rand(rng, t, 2, 3), rand(rng, t, 1, 3), rand(rng, t, 1, 3)
        do = rand(rng, t, 2, 3)
        dq, dk, dv = bwd.attention_backward_varlen(q, k, v, do, cu, scale=scale, causal=causal)

        def loss(args):
            o, _ = fwd.attention_varlen(args["q"], args["k"], args["v"], cu, scale=scale,
                                        causal=causal)
            return float((o * do).sum())

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                num[idx] = (loss({"q": q, "k": k, "v": v, name: xp})
                            - loss({"q": q, "k": k, "v": v, name: xm})) / (2 * eps)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=f"varlen d{name}")


BACKWARD_PINS = [pin_backward_finite_differences, pin_backward_invariants,
                 pin_backward_dense_layout, pin_backward_varlen_finite_differences]
