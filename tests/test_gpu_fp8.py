"""GPU parity of the FP8 (e4m3) dense prefill (fa_fwd_fp8).

The oracle evaluates exact attention on the dequantised inputs
(code * descale).  The kernel rounds the softmax weights P to e4m3 before
the P V product, so two kinds of check are used:

* exact-P inputs (integer base-2 scores, so every weight is a power of two
  and exact in e4m3): the bf16 tolerance of the other prefill tests;
* N(0, 1) inputs quantised per tensor: a per-element bound derived from the
  e4m3 rounding, |p~ - p| <= 2^-4 p + 2^-10 (3 mantissa bits; spacing 2^-9
  below 2^-6), with p = exp(s - m) relative to the row maximum m (the
  kernel's reference maximum never exceeds m, so its weights are rounded at
  least this finely):
      |o - o*| <= 2^-4 * attn(|v|) + 2^-10 * sum_j |v_j| / l + 2^-8 |o*| + 1e-4
  where attn(|v|) is the oracle's output for |v|, l = exp(lse* - m) and the
  2^-8 term covers the bf16 output.  The weights' rounding errors are
  independent of v, so the relative RMS error over all entries is about
  2^-4 / sqrt(3) = 0.036; the test allows 0.05.  The scores are products of
  e4m3 values accumulated in fp32, so the LSE keeps the 1e-3 tolerance.
"""
import math

import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import TOL_LSE, assert_device_clean, compare, host_f64, torch_mod

pytestmark = pytest.mark.gpu

REL_RMS_MAX = 0.05


@pytest.fixture(scope="module")
def fa():
    from exact_attention_33_gb300.build import build
    build()
    import exact_attention_33_gb300 as fa_mod
    fa_mod.fa_device_status(clear=True)
    return fa_mod


def dev_u8(codes):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).cuda()


def run_fp8(fa, inp, causal):
    torch = torch_mod()
    out, lse = fa.fa_fwd_fp8(dev_u8(inp.q), dev_u8(inp.k), dev_u8(inp.v), inp.q_descale,
                             inp.k_descale, inp.v_descale, causal=causal, scale=inp.scale)
    torch.cuda.synchronize()
    return host_f64(out), lse.cpu().numpy().astype(np.float64)


def row_max_scores(q, k, scale, causal, rows):
    """max_j scale * q_i . k_j over the visible keys of each listed row.
    q: [N, d] (one head), k: [N, d]; returns [len(rows)]."""
    s = scale * (q[rows] @ k.T)
    if causal:
        s = np.where(np.arange(k.shape[0])[None, :] <= np.asarray(rows)[:, None], s, -np.inf)
    return s.max(axis=1)


def check_bound(out, q, k, v, scale, causal, o_ref, lse_ref, rows, what):
    """Per-element e4m3 bound for one head; q [N, d], k/v [N, d], out and
    o_ref [len(rows), d], lse_ref [len(rows)]."""
    o_abs, _ = oracle.attention_one(q[:, None], k[:, None], np.abs(v)[:, None], scale=scale,
                                    causal=causal, rows=rows)
    o_abs = o_abs[:, 0]
    m = row_max_scores(q, k, scale, causal, rows)
    cum_abs = np.cumsum(np.abs(v), axis=0)
    vis_abs = cum_abs[np.asarray(rows)] if causal else np.broadcast_to(cum_abs[-1], o_ref.shape)
    inv_l = np.exp(m - lse_ref)[:, None]
    bound = 2.0 ** -4 * o_abs + 2.0 ** -10 * vis_abs * inv_l + 2.0 ** -8 * np.abs(o_ref) + 1e-4
    err = np.abs(out - o_ref)
    worst = float((err / bound).max())
    assert worst <= 1.0, f"{what}: error reaches {worst:.3f} of the e4m3 bound"
    return err


def check_random(out, lse, inp, causal, o_ref, l_ref, what, sample=None):
    """Bound per element and relative RMS over all checked entries."""
    scale = inp.scale if inp.scale is not None else 1.0 / math.sqrt(inp.d)
    q, k, v = inp.real("q"), inp.real("k"), inp.real("v")
    group = inp.H // inp.Hkv
    errs, refs = [], []
    pairs = sample if sample is not None else [(b, h) for b in range(inp.B) for h in range(inp.H)]
    for b, h in pairs:
        g = h // group
        rows = np.arange(inp.N)
        o_bh = o_ref[(b, h)] if isinstance(o_ref, dict) else o_ref[b, :, h]
        l_bh = l_ref[(b, h)] if isinstance(l_ref, dict) else l_ref[b, h]
        errs.append(check_bound(out[b, :, h], q[b, :, h], k[b, :, g], v[b, :, g], scale, causal,
                                o_bh, l_bh, rows, f"{what} b{b} h{h}"))
        refs.append(o_bh)
        fin = np.isfinite(l_bh)
        lerr = float(np.abs(lse[b, h][fin] - l_bh[fin]).max()) if fin.any() else 0.0
        assert lerr <= TOL_LSE, f"{what} b{b} h{h}: max |lse err| {lerr:.3e}"
    err = np.concatenate([e.reshape(-1) for e in errs])
    ref = np.concatenate([r.reshape(-1) for r in refs])
    rel = math.sqrt(float(np.mean(err ** 2)) / max(float(np.mean(ref ** 2)), 1e-30))
    assert rel <= REL_RMS_MAX, f"{what}: relative RMS error {rel:.4f} > {REL_RMS_MAX}"
    return rel


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,H,Hkv", [(1, 2, 1), (100, 2, 1), (300, 4, 4), (1000, 4, 2),
                                     (2500, 2, 1)])
def test_fp8_exact_weights(fa, causal, N, H, Hkv, d):
    """Powers-of-two weights: the e4m3 P is exact, so the bf16 bar applies.
    At d = 64 an e4m3 row is 64 bytes (the 64-byte swizzle)."""
    inp = W.fp8_exact_p_inputs(1, N, H, Hkv, d, seed=N + H + d)
    out, lse = run_fp8(fa, inp, causal)
    o_ref, l_ref = oracle.attention_dense(inp.real("q"), inp.real("k"), inp.real("v"),
                                          scale=inp.scale, causal=causal)
    compare(out, o_ref, lse, l_ref, f"fp8 exact N{N} H{H}/{Hkv} d{d} causal={causal}")
    assert_device_clean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,N,H,Hkv", [(1, 200, 2, 1), (2, 777, 4, 2), (1, 1500, 2, 2)])
def test_fp8_random(fa, causal, B, N, H, Hkv, d):
    inp = W.fp8_inputs(B, N, H, Hkv, d, seed=40 + N + d)
    out, lse = run_fp8(fa, inp, causal)
    o_ref, l_ref = oracle.attention_dense(inp.real("q"), inp.real("k"), inp.real("v"),
                                          causal=causal)
    rel = check_random(out, lse, inp, causal, o_ref, l_ref, f"fp8 N{N} d{d} causal={causal}")
    print(f"fp8 N{N} B{B} H{H}/{Hkv} d{d} causal={causal}: relative RMS error {rel:.4f}")
    assert_device_clean()


def test_fp8_descales_enter_linearly(fa):
    """Scaling a descale by 2 scales the scores (q, k) or the output (v)."""
    inp = W.fp8_exact_p_inputs(1, 300, 2, 1, 128, seed=3)
    base, lse_base = run_fp8(fa, inp, True)
    inp.v_descale *= 2.0
    out_v, lse_v = run_fp8(fa, inp, True)
    assert np.allclose(out_v, 2.0 * base, rtol=0, atol=0)
    assert np.array_equal(lse_v, lse_base)
    rnd = W.fp8_inputs(1, 600, 2, 1, 128, seed=12)
    rnd.q_descale *= 2.0
    rnd.k_descale *= 0.5 ** 3
    out_q, lse_q = run_fp8(fa, rnd, True)
    o_ref, l_ref = oracle.attention_dense(rnd.real("q"), rnd.real("k"), rnd.real("v"),
                                          causal=True)
    check_random(out_q, lse_q, rnd, True, o_ref, l_ref, "fp8 q x2 k /8")
    assert_device_clean()


def test_fp8_full_size_sampled(fa):
    """The FP8 causal workload at full size (B=2, H=32, N=8192, d=128); the
    oracle evaluates 3 seeded (batch, head) pairs."""
    cfg = W.WORKLOADS["long_causal_fp8_d128"]
    inp = W.fp8_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    out, lse = run_fp8(fa, inp, True)
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(9)
    pairs = [(int(x) // inp.H, int(x) % inp.H) for x in rng.choice(inp.B * inp.H, 3, replace=False)]
    o_ref, l_ref = {}, {}
    for b, h in pairs:
        o1, l1 = oracle.attention_one(inp.real("q")[b][:, h:h + 1], inp.real("k")[b][:, h:h + 1],
                                      inp.real("v")[b][:, h:h + 1], causal=True)
        o_ref[(b, h)], l_ref[(b, h)] = o1[:, 0], l1[0]
    rel = check_random(out, lse, inp, True, o_ref, l_ref, "fp8 full", sample=pairs)
    print(f"fp8 full size sampled: relative RMS error {rel:.4f}")
    assert_device_clean()


def test_fp8_deterministic_and_rejects(fa):
    torch = torch_mod()
    inp = W.fp8_inputs(1, 500, 2, 1, 128, seed=11)
    q, k, v = dev_u8(inp.q), dev_u8(inp.k), dev_u8(inp.v)
    o1, l1 = fa.fa_fwd_fp8(q, k, v, 1.0, 1.0, 1.0, causal=True)
    o2, l2 = fa.fa_fwd_fp8(q, k, v, 1.0, 1.0, 1.0, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    q96 = torch.zeros((1, 8, 2, 96), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_fp8(q96, q96, q96, 1.0, 1.0, 1.0)
    assert e.value.status == -2
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_fp8(q, k, v, 1.0, 0.0, 1.0)
    assert e.value.status == -1


# ---------------------------------------------------------------- packed varlen

def varlen_fp8_case(inp, lengths):
    """The tokens of a B = 1 FP8 input cut into sequences of ``lengths``."""
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    assert cu[-1] == inp.N
    return cu


def run_varlen_fp8(fa, inp, cu, causal):
    torch = torch_mod()
    dev_cu = torch.from_numpy(cu).cuda()
    out, lse = fa.fa_fwd_varlen_fp8(dev_u8(inp.q[0]), dev_u8(inp.k[0]), dev_u8(inp.v[0]), dev_cu,
                                    int(np.diff(cu).max()), inp.q_descale, inp.k_descale,
                                    inp.v_descale, causal=causal, scale=inp.scale)
    torch.cuda.synchronize()
    return host_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (3, 1)])   # head pairs, and row pairs (odd group)
def test_fp8_varlen_exact_weights(fa, causal, H, Hkv, d):
    """Packed sequences (ragged, one empty, one of a single token) with
    powers-of-two weights: the bf16 bar applies."""
    lengths = [300, 1, 0, 129, 640, 77]
    inp = W.fp8_exact_p_inputs(1, sum(lengths), H, Hkv, d, seed=31 + H + d)
    cu = varlen_fp8_case(inp, lengths)
    out, lse = run_varlen_fp8(fa, inp, cu, causal)
    o_ref, l_ref = oracle.attention_varlen(inp.real("q")[0], inp.real("k")[0], inp.real("v")[0],
                                           cu, scale=inp.scale, causal=causal)
    compare(out, o_ref, lse, l_ref, f"fp8 varlen exact H{H}/{Hkv} d{d} causal={causal}")
    assert_device_clean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (3, 1)])
def test_fp8_varlen_random(fa, H, Hkv, d):
    """N(0, 1) inputs quantised per tensor, causal: the e4m3 bound of
    check_bound per sequence and head, and the relative RMS over all."""
    lengths = [517, 64, 1300, 200]
    inp = W.fp8_inputs(1, sum(lengths), H, Hkv, d, seed=55 + H + d)
    cu = varlen_fp8_case(inp, lengths)
    out, lse = run_varlen_fp8(fa, inp, cu, True)
    q, k, v = inp.real("q")[0], inp.real("k")[0], inp.real("v")[0]
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, causal=True)
    scale = 1.0 / math.sqrt(d)
    group = H // Hkv
    errs, refs = [], []
    for s in range(len(lengths)):
        a, e = int(cu[s]), int(cu[s + 1])
        rows = np.arange(e - a)
        for h in range(H):
            g = h // group
            errs.append(check_bound(out[a:e, h], q[a:e, h], k[a:e, g], v[a:e, g], scale, True,
                                    o_ref[a:e, h], l_ref[h, a:e], rows, f"fp8 varlen s{s} h{h}"))
            refs.append(o_ref[a:e, h])
    lerr = float(np.abs(lse - l_ref).max())
    assert lerr <= TOL_LSE, f"fp8 varlen: max |lse err| {lerr:.3e}"
    err = np.concatenate([x.reshape(-1) for x in errs])
    ref = np.concatenate([x.reshape(-1) for x in refs])
    rel = math.sqrt(float(np.mean(err ** 2)) / max(float(np.mean(ref ** 2)), 1e-30))
    assert rel <= REL_RMS_MAX, f"fp8 varlen: relative RMS error {rel:.4f} > {REL_RMS_MAX}"
    assert_device_clean()
