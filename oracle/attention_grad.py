"""fp64 CPU oracle for the gradient of exact attention (backward pass).

TEST INFRASTRUCTURE ONLY, like ``oracle.attention``: nothing in the product
path imports or runs it, and it shares no code with the CUDA library.

The pages describe only the forward computation (the streaming softmax); they
say that the method trains models but give no backward algorithm.  What the
backward pass must return is nevertheless fixed by the forward definition:
the gradient of a loss through O = softmax(scale * Q K^T) V, with the causal
and GQA conventions of ``oracle.attention``.  For one (sequence, query head)
with upstream gradient dO, the chain rule gives (P the attention weights,
masked entries 0):

    dV = P^T dO                                   (O = P V)
    dP = dO V^T
    dS_ij = P_ij (dP_ij - D_i),  D_i = sum_j P_ij dP_ij = sum_c dO_ic O_ic
                                                  (row-wise softmax)
    dQ = scale * dS K,   dK = scale * dS^T Q      (S = scale Q K^T)

A key/value head receives the sum over the query heads that read it.  The
log-sum-exp is an output of the forward pass but no gradient flows through it
here (dLSE = 0).  Rows with no visible key have P = 0 and contribute nothing.

Pinned in ``tests/oracle_pins.py`` by central finite differences of the
scalar <O, dO> on tiny inputs (independent of these formulas), and by the
invariants sum_j dV_j = sum_i dO_i (rows of P sum to 1) and, without a
mask, sum_j dK_j = 0 (softmax is unchanged when every key moves by the same
vector).  The packed (varlen) form is pinned by finite differences through
the packed forward oracle ``oracle.attention.attention_varlen``.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["attention_backward_one", "attention_backward_dense", "attention_backward_varlen"]


def attention_backward_one(q, k, v, do, scale=None, causal=False):
    """Gradients of one sequence, all heads.

    q, do: [Nq, H, d]; k, v: [Nk, Hkv, d].  Returns (dq [Nq, H, d],
    dk [Nk, Hkv, d], dv [Nk, Hkv, d]) in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    nq, h_q, d = q.shape
    nk, h_kv, _ = k.shape
    if h_q % h_kv != 0:
        raise ValueError("H must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = h_q // h_kv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if nq == 0 or nk == 0:
        return dq, dk, dv
    if causal:
        visible = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
    else:
        visible = np.ones((nq, nk), dtype=bool)
    for h in range(h_q):
        g = h // group
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1)
        live = np.isfinite(m)
        e = np.exp(s - np.where(live, m, 0.0)[:, None])
        z = e.sum(axis=1)
        p = np.divide(e, z[:, None], out=np.zeros_like(e), where=live[:, None])
        o = p @ v[:, g, :]
        dv[:, g, :] += p.T @ do[:, h, :]
        dp = do[:, h, :] @ v[:, g, :].T
        d_row = (do[:, h, :] * o).sum(axis=1)
        ds = p * (dp - d_row[:, None])
        dq[:, h, :] = scale * (ds @ k[:, g, :])
        dk[:, g, :] += scale * (ds.T @ q[:, h, :])
    return dq, dk, dv


def attention_backward_dense(q, k, v, do, scale=None, causal=False):
    """Batched dense layout: q, do [B, N, H, d]; k, v [B, N, Hkv, d]."""
    outs = [attention_backward_one(q[b], k[b], v[b], do[b], scale=scale, causal=causal)
            for b in range(np.asarray(q).shape[0])]
    return tuple(np.stack([o[i] for o in outs]) for i in range(3))


def attention_backward_varlen(q, k, v, do, cu_seqlens, scale=None, causal=False):
    """Packed variable-length batch (the explainer article's "Varlen" section):
    q, do [T, H, d]; k, v [T, Hkv, d]; sequence s owns rows [cu[s], cu[s+1])
    and sees only its own keys, so its gradients are those of the sequence on
    its own.  Rows outside every sequence get zero gradients."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        dq[a:e], dk[a:e], dv[a:e] = attention_backward_one(q[a:e], k[a:e], v[a:e], do[a:e],
                                                           scale=scale, causal=causal)
    return dq, dk, dv
