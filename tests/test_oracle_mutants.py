"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (the mistakes live only here, on the CPU)."""
import math

import numpy as np
import pytest

import oracle.attention as ora_mod
from oracle_pins import ALL_PINS


def mutant_attention_one(mistake):
    def attention_one(q, k, v, scale=None, causal=False, rows=None, heads=None):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        nq, h_q, d = q.shape
        nk, h_kv, _ = k.shape
        if scale is None:
            scale = 1.0 / math.sqrt(d) if mistake != "default_scale_1_over_d" else 1.0 / d
        if mistake == "no_scale":
            scale = 1.0
        group = h_q // h_kv
        o = np.zeros((nq, h_q, v.shape[2]))
        lse = np.full((h_q, nq), -np.inf)
        sel = np.arange(nq)
        cols = np.arange(nk)[None, :]
        if causal:
            off = 0 if mistake == "top_left_causal" else (nk - nq)
            visible = cols <= sel[:, None] + off
            if mistake == "causal_off_by_one":
                visible = cols < sel[:, None] + off
        else:
            visible = np.ones((nq, nk), dtype=bool)
        for h in range(h_q):
            g = h % h_kv if mistake == "gqa_modulo" else h // group
            s = scale * (q[:, h, :] @ k[:, g, :].T)
            if mistake == "sign":
                s = -s
            s = np.where(visible, s, -np.inf)
            mx = s.max(axis=1)
            live = np.isfinite(mx)
            mx0 = np.where(live, mx, 0.0)
            e = np.exp(s - mx0[:, None])
            z = e.sum(axis=1)
            p = np.divide(e, z[:, None], out=np.zeros_like(e), where=live[:, None])
            vals = k if mistake == "keys_as_values" else v
            o[:, h, :] = p @ vals[:, g, :v.shape[2]] if mistake != "keys_as_values" else p @ vals[:, g, :]
            if mistake == "lse_no_max":
                lse[h] = np.where(live, np.log(np.where(live, z, 1.0)), -np.inf)
            elif mistake == "lse_log2":
                lse[h] = np.where(live, mx0 + np.log2(np.where(live, z, 1.0)), -np.inf)
            else:
                lse[h] = np.where(live, mx0 + np.log(np.where(live, z, 1.0)), -np.inf)
        return o, lse
    return attention_one


def mutant_merge_no_rescale(states):
    states = list(states)
    m = max(s[0] for s in states)
    return m, sum(s[1] for s in states), sum(np.asarray(s[2], dtype=np.float64) for s in states)


def mutant_tile_state_no_max(scores, values=None):
    s = np.asarray(scores, dtype=np.float64).reshape(-1)
    vals = np.zeros((s.shape[0], 0)) if values is None else np.asarray(values).reshape(s.shape[0], -1)
    if s.size == 0:
        return -np.inf, 0.0, np.zeros(vals.shape[1])
    w = np.exp(s)
    return float(s.max()), float(w.sum()), w @ vals


def mutant_gather_whole_last_block(pool, row, ctx_len, block_size):
    n_blocks = (int(ctx_len) + block_size - 1) // block_size
    return np.concatenate([np.asarray(pool)[int(row[i])] for i in range(n_blocks)], axis=0)


def mutant_varlen_leak(q, k, v, cu_seqlens, scale=None, causal=False):
    o, lse = ora_mod.attention_one(q, k, v, scale=scale, causal=causal)
    return o, lse


ATTN_MISTAKES = ["no_scale", "default_scale_1_over_d", "top_left_causal", "causal_off_by_one",
                 "gqa_modulo", "sign", "keys_as_values", "lse_no_max", "lse_log2"]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(ora_mod, name, fn)
    failures = 0
    for pin in ALL_PINS:
        try:
            pin(ora_mod)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    return failures


@pytest.mark.parametrize("mistake", ATTN_MISTAKES)
def test_attention_mistake_is_caught(monkeypatch, mistake):
    assert _caught(monkeypatch, "attention_one", mutant_attention_one(mistake)) > 0


@pytest.mark.parametrize("name,fn", [
    ("merge_states", mutant_merge_no_rescale),
    ("tile_state", mutant_tile_state_no_max),
    ("gather_paged", mutant_gather_whole_last_block),
    ("attention_varlen", mutant_varlen_leak),
])
def test_helper_mistake_is_caught(monkeypatch, name, fn):
    assert _caught(monkeypatch, name, fn) > 0


def test_unmutated_oracle_passes_all_pins():
    for pin in ALL_PINS:
        pin(ora_mod)


# ------------------------------------------------------------ backward pass
import oracle.attention_grad as grad_mod  # noqa: E402
from oracle_pins import BACKWARD_PINS  # noqa: E402


def mutant_backward_one(mistake):
    def attention_backward_one(q, k, v, do, scale=None, causal=False):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        nq, h_q, d = q.shape
        nk, h_kv, _ = k.shape
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        group = h_q // h_kv
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        if causal:
            visible = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
        else:
            visible = np.ones((nq, nk), dtype=bool)
        for h in range(h_q):
            g = h // group
            s = np.where(visible, scale * (q[:, h] @ k[:, g].T), -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            p = e / e.sum(axis=1)[:, None]
            o = p @ v[:, g]
            if mistake == "dv_no_transpose":
                dv[:, g] += (p @ do[:, h])[:nk] if nq >= nk else np.pad(p @ do[:, h], ((0, nk - nq), (0, 0)))
            else:
                dv[:, g] += p.T @ do[:, h]
            dp = do[:, h] @ v[:, g].T
            d_row = 0.0 if mistake == "no_d_term" else (do[:, h] * o).sum(axis=1)[:, None]
            ds = p * (dp - d_row)
            sc = 1.0 if mistake == "dq_no_scale" else scale
            dq[:, h] = sc * (ds @ k[:, g])
            if mistake == "dk_overwrite_group":
                dk[:, g] = scale * (ds.T @ q[:, h])
            elif mistake == "dk_sign":
                dk[:, g] -= scale * (ds.T @ q[:, h])
            else:
                dk[:, g] += scale * (ds.T @ q[:, h])
        return dq, dk, dv
    return attention_backward_one


@pytest.mark.parametrize("mistake", ["dv_no_transpose", "no_d_term", "dq_no_scale",
                                     "dk_overwrite_group", "dk_sign"])
def test_backward_mistake_is_caught(monkeypatch, mistake):
    monkeypatch.setattr(grad_mod, "attention_backward_one", mutant_backward_one(mistake))
    failures = 0
    for pin in BACKWARD_PINS:
        try:
            pin(ora_mod, grad_mod)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0


def mutant_backward_varlen(mistake):
    one = grad_mod.attention_backward_one

    def attention_backward_varlen(q, k, v, do, cu_seqlens, scale=None, causal=False):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        if mistake == "one_sequence":  # keys seen across sequence boundaries
            return one(q, k, v, do, scale=scale, causal=causal)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for s in range(len(cu) - 1):
            a, e = int(cu[s]), int(cu[s + 1])
            if mistake == "keys_from_start":  # every sequence reads the first keys
                r = one(q[a:e], k[:e - a], v[:e - a], do[a:e], scale=scale, causal=causal)
            else:  # "last_row_dropped"
                r = one(q[a:max(a, e - 1)], k[a:e], v[a:e], do[a:max(a, e - 1)], scale=scale,
                        causal=causal)
                r = (np.concatenate([r[0], np.zeros((e - a - r[0].shape[0],) + q.shape[1:])]),
                     r[1], r[2])
            dq[a:e], dk[a:e], dv[a:e] = r
        return dq, dk, dv
    return attention_backward_varlen


@pytest.mark.parametrize("mistake", ["one_sequence", "keys_from_start", "last_row_dropped"])
def test_backward_varlen_mistake_is_caught(monkeypatch, mistake):
    monkeypatch.setattr(grad_mod, "attention_backward_varlen", mutant_backward_varlen(mistake))
    failures = 0
    for pin in BACKWARD_PINS:
        try:
            pin(ora_mod, grad_mod)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0
