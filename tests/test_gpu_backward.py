"""GPU parity of the backward pass (fa_bwd) against the fp64 gradient oracle.

The kernel takes the bf16 output and fp32 log-sum-exp of fa_fwd, recomputes
the weights P in fp32, and rounds P and dS to bf16 for the tensor-core
products (fp32 accumulation); D = rowsum(dO * O) is formed from the bf16 O;
the three gradients are written in bf16.  Each of those roundings moves an
element by at most 2^-9 of its size.  Five such steps, with independent
errors, give a relative RMS error near 5 * 2^-9 / sqrt(3) = 5.6e-3 per
gradient tensor; the test allows REL_RMS_MAX = 1.5e-2.  Element-wise, an
error of a few of those roundings of the largest terms is allowed:
|err| <= MAX_OVER_MAX * max|reference| (the scale of the gradient rows varies
widely under a causal mask, so the tensor's RMS is not the reference here).
"""
import math

import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import assert_device_clean, dev_bf16, dev_i32, host_f64, torch_mod

pytestmark = pytest.mark.gpu

REL_RMS_MAX = 1.5e-2
MAX_OVER_MAX = 2e-2


@pytest.fixture(scope="module")
def fa():
    from exact_attention_33_gb300.build import build
    build()
    import exact_attention_33_gb300 as fa_mod
    fa_mod.fa_device_status(clear=True)
    return fa_mod


def f64(bits):
    return W.bf16_bits_to_f64(bits)


def check_grad(name, got, ref, what):
    err = got - ref
    rms = math.sqrt(float(np.mean(ref ** 2))) if ref.size else 0.0
    if rms < 1e-12:
        # an exactly-zero gradient (a single visible key: dS = P (dP - D) with
        # dP and D the same dot product summed in two orders) is met to
        # fp32 reassociation error
        assert float(np.abs(got).max()) <= 1e-4, f"{what} {name}: nonzero where the gradient is 0"
        return 0.0
    rel = math.sqrt(float(np.mean(err ** 2))) / rms
    mx = float(np.abs(err).max()) / float(np.abs(ref).max())
    assert np.all(np.isfinite(got)), f"{what} {name}: non-finite values"
    assert rel <= REL_RMS_MAX, f"{what} {name}: relative RMS error {rel:.3e}"
    assert mx <= MAX_OVER_MAX, f"{what} {name}: max error {mx:.3e} of the largest gradient"
    return rel


def run_case(fa, B, N, H, Hkv, d, causal, seed, scale=None):
    torch = torch_mod()
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=seed)
    do_bits = W.normal_bf16_bits((B, N, H, d), seed, 3)
    q, k, v, do = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_bf16(do_bits)
    out, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, out, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attention_backward_dense(f64(inp.q), f64(inp.k), f64(inp.v), f64(do_bits),
                                                 scale=scale, causal=causal)
    what = f"B{B} N{N} H{H}/{Hkv} d{d} causal={causal}"
    errs = [check_grad(n, host_f64(g), r, what) for n, g, r in
            (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv))]
    print(f"{what}: relative RMS errors dq {errs[0]:.2e} dk {errs[1]:.2e} dv {errs[2]:.2e}")
    assert_device_clean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,N,H,Hkv", [(1, 1, 2, 1), (1, 100, 2, 1), (2, 128, 2, 2),
                                       (1, 300, 4, 2), (1, 777, 2, 1)])
def test_backward_small(fa, d, causal, B, N, H, Hkv):
    run_case(fa, B, N, H, Hkv, d, causal, seed=90 + N)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_wide_group(fa, causal):
    """Eight query heads per KV head: each dK/dV item runs 8 iterations per
    query tile and sums the whole group in TMEM."""
    run_case(fa, 1, 300, 8, 1, 128, causal, seed=98)


def test_backward_medium(fa):
    """Many tiles in both directions (16 query and 16 key tiles)."""
    run_case(fa, 1, 2048, 2, 1, 128, True, seed=95)


def test_backward_explicit_scale(fa):
    run_case(fa, 1, 260, 2, 2, 64, False, seed=96, scale=0.3)


def test_backward_deterministic_and_rejects(fa):
    torch = torch_mod()
    inp = W.dense_inputs(1, 500, 4, 2, 128, seed=97)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    do = dev_bf16(W.normal_bf16_bits((1, 500, 4, 128), 97, 3))
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    a = fa.fa_bwd(q, k, v, out, lse, do, causal=True)
    b = fa.fa_bwd(q, k, v, out, lse, do, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(q, k, v, out, lse, do, causal=True, workspace=small)
    assert e.value.status == -4
    assert_device_clean()


def test_backward_full_size_sampled(fa):
    """The backward leg's launch at full size (the long causal workload:
    B=2, H=32, N=8192, d=128, 1% x8 key outliers).  The oracle evaluates the
    gradients of two seeded (batch, head) pairs: dQ on 256 seeded rows, dK and
    dV on 256 seeded keys (their columns of P need every row's log-sum-exp,
    so the pair's full forward runs in fp64)."""
    torch = torch_mod()
    cfg = W.WORKLOADS["long_causal_d128"]
    B, N, H, d = cfg["B"], cfg["N"], cfg["H"], cfg["d"]
    inp = W.dense_inputs(B, N, H, cfg["Hkv"], d, seed=0, outlier_frac=cfg["outlier_frac"],
                         outlier_scale=cfg["outlier_scale"])
    do_bits = W.normal_bf16_bits((B, N, H, d), 0, 3)
    q, k, v, do = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_bf16(do_bits)
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa.fa_bwd(q, k, v, out, lse, do, causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    pairs = [(int(x) // H, int(x) % H) for x in rng.choice(B * H, 2, replace=False)]
    scale = 1.0 / math.sqrt(d)
    for b, h in pairs:
        qh, kh, vh = f64(inp.q[b, :, h]), f64(inp.k[b, :, h]), f64(inp.v[b, :, h])
        doh = f64(do_bits[b, :, h])
        # the pair's forward in fp64, one block of rows at a time
        o = np.zeros((N, d))
        lse_ref = np.zeros(N)
        for r0 in range(0, N, 1024):
            o_blk, l_blk = oracle.attention_one(qh[:, None], kh[:, None], vh[:, None], causal=True,
                                                rows=np.arange(r0, min(N, r0 + 1024)))
            o[r0:r0 + 1024] = o_blk[r0:r0 + 1024, 0]
            lse_ref[r0:r0 + 1024] = l_blk[0, r0:r0 + 1024]
        dsum = (doh * o).sum(axis=1)
        rows = np.sort(rng.choice(N, 256, replace=False))
        keys = np.sort(rng.choice(N, 256, replace=False))
        # dQ rows: dS_i = P_i (dP_i - D_i), dQ_i = scale dS_i K
        s_rows = scale * (qh[rows] @ kh.T)
        s_rows[np.arange(N)[None, :] > rows[:, None]] = -np.inf
        p_rows = np.exp(s_rows - lse_ref[rows, None])
        ds_rows = p_rows * (doh[rows] @ vh.T - dsum[rows, None])
        dq_ref = scale * (ds_rows @ kh)
        # dK / dV keys: columns of P over every query
        s_cols = scale * (qh @ kh[keys].T)
        s_cols[np.arange(N)[:, None] < keys[None, :]] = -np.inf
        p_cols = np.exp(s_cols - lse_ref[:, None])
        dv_ref = p_cols.T @ doh
        ds_cols = p_cols * (doh @ vh[keys].T - dsum[:, None])
        dk_ref = scale * (ds_cols.T @ qh)
        what = f"full b{b} h{h}"
        errs = [check_grad("dq", host_f64(dq[b, rows, h]), dq_ref, what),
                check_grad("dk", host_f64(dk[b, keys, h]), dk_ref, what),
                check_grad("dv", host_f64(dv[b, keys, h]), dv_ref, what)]
        print(f"{what}: relative RMS errors dq {errs[0]:.2e} dk {errs[1]:.2e} dv {errs[2]:.2e}")
    assert_device_clean()


# ------------------------------------------------------------- packed batches
def run_varlen(fa, lengths, H, Hkv, d, causal, seed, pad_rows=0, max_seqlen=None):
    """fa_bwd_varlen on a packed batch against the packed gradient oracle,
    one sequence at a time (each sequence's gradients at the tolerance of
    its own scale).  ``pad_rows`` extra rows after the last sequence belong
    to no sequence: their gradients keep the value they had before the call."""
    torch = torch_mod()
    inp = W.varlen_inputs(lengths, H, Hkv, d, seed=seed)
    T = inp.total_tokens
    cu = inp.cu_seqlens
    max_len = int(max(lengths)) if max_seqlen is None else max_seqlen
    do_bits = W.normal_bf16_bits((T, H, d), seed, 3)
    pad = lambda bits, h: np.concatenate([bits, W.normal_bf16_bits((pad_rows, h, d), seed, 9)])
    q, k, v = dev_bf16(pad(inp.q, H)), dev_bf16(pad(inp.k, Hkv)), dev_bf16(pad(inp.v, Hkv))
    do = dev_bf16(pad(do_bits, H))
    cu_d = dev_i32(cu)
    out, lse = fa.fa_fwd_varlen(q, k, v, cu_d, max_len, causal=causal)
    sentinel = 7.0
    dq = torch.full_like(q, sentinel)
    dk = torch.full_like(k, sentinel)
    dv = torch.full_like(v, sentinel)
    fa.fa_bwd_varlen(q, k, v, out, lse, do, cu_d, max_len, causal=causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attention_backward_varlen(f64(inp.q), f64(inp.k), f64(inp.v),
                                                  f64(do_bits), cu, causal=causal)
    gq, gk, gv = host_f64(dq), host_f64(dk), host_f64(dv)
    worst = 0.0
    for s in range(len(lengths)):
        a, e = int(cu[s]), int(cu[s + 1])
        if e == a:
            continue
        what = f"seq {s} of {list(lengths)} H{H}/{Hkv} d{d} causal={causal}"
        for n, g, r in (("dq", gq, rq), ("dk", gk, rk), ("dv", gv, rv)):
            worst = max(worst, check_grad(n, g[a:e], r[a:e], what))
    if pad_rows:
        for n, g in (("dq", gq), ("dk", gk), ("dv", gv)):
            assert np.all(g[T:] == sentinel), f"{n}: a row outside every sequence was written"
    print(f"{list(lengths)} H{H}/{Hkv} d{d} causal={causal}: worst relative RMS {worst:.2e}")
    assert_device_clean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lengths,H,Hkv", [([1, 130, 0, 257, 64], 4, 2),
                                           ([300, 5, 128], 3, 1),
                                           ([129], 2, 2)])
def test_backward_varlen(fa, d, causal, lengths, H, Hkv):
    run_varlen(fa, lengths, H, Hkv, d, causal, seed=200 + sum(lengths))


def test_backward_varlen_rows_outside_sequences(fa):
    run_varlen(fa, [70, 190], 2, 1, 128, True, seed=211, pad_rows=37)


def test_backward_varlen_many_tiles(fa):
    """Sequences of 1000 to 2100 rows (8 to 17 tiles each way)."""
    run_varlen(fa, [1000, 2100, 1537], 4, 1, 128, True, seed=212)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_varlen_many_sequences(fa, causal):
    """More sequences (150) than the longest-first order covers: the tiles are
    claimed sequence by sequence, past each sequence's end claimed again."""
    lengths = np.random.default_rng(215).integers(0, 300, size=150)
    run_varlen(fa, list(lengths), 2, 1, 64, causal, seed=215)


def test_backward_varlen_loose_max_seqlen(fa):
    """A max_seqlen far above the longest sequence (levels with no tile)."""
    run_varlen(fa, [100, 37, 260], 4, 2, 128, True, seed=216, max_seqlen=1000)


def test_backward_varlen_matches_dense(fa):
    """Equal lengths packed back to back give the dense call's gradients bit
    for bit (the same tiles in the same order)."""
    torch = torch_mod()
    B, N, H, Hkv, d = 3, 200, 4, 2, 64
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=213)
    do_bits = W.normal_bf16_bits((B, N, H, d), 213, 3)
    q, k, v, do = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_bf16(do_bits)
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    dense = fa.fa_bwd(q, k, v, out, lse, do, causal=True)
    cu = dev_i32(np.arange(B + 1) * N)
    flat = lambda t: t.reshape(B * N, t.shape[2], d)
    packed = fa.fa_bwd_varlen(flat(q), flat(k), flat(v), flat(out),
                              lse.permute(1, 0, 2).reshape(H, B * N).contiguous(), flat(do), cu, N,
                              causal=True)
    torch.cuda.synchronize()
    for x, y in zip(dense, packed):
        assert torch.equal(flat(x), y)
    assert_device_clean()


def test_backward_varlen_bad_cu_seqlens_flagged(fa):
    torch = torch_mod()
    inp = W.varlen_inputs([10, 20], 2, 2, 64, seed=214)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    cu = dev_i32(inp.cu_seqlens)
    out, lse = fa.fa_fwd_varlen(q, k, v, cu, 20)
    torch.cuda.synchronize()
    fa.fa_device_status(clear=True)
    for bad, max_len in (([0, 25, 20], 25), ([0, 10, 30], 15)):   # decreasing; too long
        fa.fa_bwd_varlen(q, k, v, out, lse, q, dev_i32(np.array(bad, dtype=np.int32)), max_len)
        torch.cuda.synchronize()
        assert fa.fa_device_status(clear=True) & fa.FA_DEV_BAD_SEQLEN
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_varlen(q, k, v, out, lse, q, cu, 20, workspace=small)
    assert e.value.status == -4
    assert_device_clean()


def test_backward_varlen_full_size_sampled(fa):
    """The packed backward leg's launch at full size (the varlen workload: 32
    sequences of U[64, 4096] tokens, H 16 / Hkv 4, d 128, causal).  The
    oracle computes the full gradients of two seeded (sequence, KV group)
    slices (the group's 4 query heads), which are compared with the kernels'."""
    torch = torch_mod()
    cfg = W.WORKLOADS["varlen_gqa_d128"]
    lengths = W.varlen_lengths(cfg["num_seqs"], cfg["len_lo"], cfg["len_hi"])
    H, Hkv, d = cfg["H"], cfg["Hkv"], cfg["d"]
    inp = W.varlen_inputs(lengths, H, Hkv, d, seed=0)
    T = inp.total_tokens
    do_bits = W.normal_bf16_bits((T, H, d), 0, 3)
    q, k, v, do = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_bf16(do_bits)
    cu = dev_i32(inp.cu_seqlens)
    max_len = int(np.max(lengths))
    out, lse = fa.fa_fwd_varlen(q, k, v, cu, max_len, causal=True)
    dq, dk, dv = fa.fa_bwd_varlen(q, k, v, out, lse, do, cu, max_len, causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(17)
    group = H // Hkv
    for s in rng.choice(len(lengths), 2, replace=False):
        g = int(rng.integers(0, Hkv))
        a, e = int(inp.cu_seqlens[s]), int(inp.cu_seqlens[s + 1])
        hs = slice(g * group, (g + 1) * group)
        rq, rk, rv = oracle.attention_backward_one(
            f64(inp.q[a:e, hs]), f64(inp.k[a:e, g:g + 1]), f64(inp.v[a:e, g:g + 1]),
            f64(do_bits[a:e, hs]), causal=True)
        what = f"full seq {s} ({e - a} rows) kv group {g}"
        errs = [check_grad("dq", host_f64(dq[a:e, hs]), rq, what),
                check_grad("dk", host_f64(dk[a:e, g:g + 1]), rk, what),
                check_grad("dv", host_f64(dv[a:e, g:g + 1]), rv, what)]
        print(f"{what}: relative RMS errors dq {errs[0]:.2e} dk {errs[1]:.2e} dv {errs[2]:.2e}")
    assert_device_clean()
