"""GPU parity of the dense prefill path (fa_fwd) against the fp64 oracle."""
import math

import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import assert_device_clean, compare, dev_bf16, host_f64, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_attention_33_gb300.build import build
    build()
    import exact_attention_33_gb300 as fa_mod
    fa_mod.fa_device_status(clear=True)
    return fa_mod


def run_dense(fa, inp, causal, scale=None):
    torch = torch_mod()
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    out, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return host_f64(out), lse.cpu().numpy().astype(np.float64)


def f64(bits):
    return W.bf16_bits_to_f64(bits)


def test_pr1_reference_case(fa):
    cfg = W.WORKLOADS["pr1"]
    inp = W.dense_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    out, lse = run_dense(fa, inp, causal=False, scale=1 / 8)
    o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), scale=1 / 8)
    compare(out, o_ref, lse, l_ref, "pr1")
    assert_device_clean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,N,H,Hkv", [(1, 1, 2, 2), (2, 77, 4, 2), (1, 128, 2, 1),
                                       (2, 300, 4, 4), (1, 513, 2, 2), (1, 1000, 8, 1)])
def test_dense_small(fa, d, causal, B, N, H, Hkv):
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=100 + N)
    out, lse = run_dense(fa, inp, causal)
    o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), causal=causal)
    compare(out, o_ref, lse, l_ref, f"dense B{B} N{N} H{H}/{Hkv} d{d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_dense_d64_config(fa, causal):
    cfg = W.WORKLOADS["dense_d64"]
    inp = W.dense_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    out, lse = run_dense(fa, inp, causal)
    o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), causal=causal)
    compare(out, o_ref, lse, l_ref, f"dense_d64 causal={causal}")
    assert_device_clean()


@pytest.fixture(scope="module")
def long_inputs():
    cfg = W.WORKLOADS["long_causal_d128"]
    return W.dense_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"], seed=0,
                          outlier_frac=cfg["outlier_frac"], outlier_scale=cfg["outlier_scale"])


def test_long_causal_config_sampled(fa, long_inputs):
    """Full-size launch; the oracle evaluates 4 seeded (batch, head) pairs."""
    inp = long_inputs
    out, lse = run_dense(fa, inp, causal=True)
    rng = np.random.default_rng(5)
    pairs = [(int(x) // inp.H, int(x) % inp.H) for x in rng.choice(inp.B * inp.H, 4, replace=False)]
    for b, h in pairs:
        g = h // (inp.H // inp.Hkv)
        o_ref, l_ref = oracle.attention_one(f64(inp.q[b][:, h:h + 1]), f64(inp.k[b][:, g:g + 1]),
                                            f64(inp.v[b][:, g:g + 1]), causal=True)
        compare(out[b, :, h], o_ref[:, 0], lse[b, h], l_ref[0], f"long b{b} h{h}")
    assert np.all(np.isfinite(out))
    assert_device_clean()


def dominant_key_inputs(N, H, d, pos, target_log2, seed):
    """Query rows close to one direction u per head, and key `pos` equal to
    c u with c chosen so that its scaled score is about `target_log2` (in
    log2 units) above the typical row maximum: one key that dominates every
    row and moves the reference maximum when its key tile arrives."""
    rng = np.random.default_rng(seed)
    u = rng.standard_normal((H, d)).astype(np.float32)
    q = (u[None, None] + 0.1 * rng.standard_normal((1, N, H, d))).astype(np.float32)
    k = rng.standard_normal((1, N, H, d)).astype(np.float32)
    v = rng.standard_normal((1, N, H, d)).astype(np.float32)
    c = target_log2 / (np.einsum("hd,hd->h", u, u) / math.sqrt(d) * math.log2(math.e))
    k[0, pos] = u * c[:, None]
    bits = W.f32_to_bf16_bits
    return W.DenseInputs(1, N, H, H, d, bits(q), bits(k), bits(v))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("pos", [10, 300, 356, 600])
@pytest.mark.parametrize("target_log2", [40.0, 200.0])
def test_dominant_key_moves_the_reference(fa, d, pos, target_log2):
    """A key far above the running maximum, in the first key tile (handled
    by that tile's maximum), in the first or second 64-key half of a later
    tile, and in the last tile.  At 40 (log2 units) its weight passes the
    lazy re-centring bound but is kept for the tile; at 200 it overflows fp32
    against the old reference, and the tile is redone (first half) or its
    stored first half rescaled (second half).  Causal and not, every element."""
    inp = dominant_key_inputs(640, 2, d, pos, target_log2, seed=41 + pos)
    for causal in (False, True):
        out, lse = run_dense(fa, inp, causal)
        o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), causal=causal)
        compare(out, o_ref, lse, l_ref, f"dominant key d{d} pos {pos} {target_log2} causal={causal}")
    assert_device_clean()


def test_deterministic(fa):
    torch = torch_mod()
    inp = W.dense_inputs(2, 700, 4, 2, 128, seed=7)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    o1, l1 = fa.fa_fwd(q, k, v, causal=True)
    o2, l2 = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_explicit_scale_and_no_lse(fa):
    torch = torch_mod()
    inp = W.dense_inputs(1, 200, 2, 2, 64, seed=8)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    out, lse = fa.fa_fwd(q, k, v, causal=False, scale=0.3, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    o_ref, _ = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), scale=0.3)
    compare(host_f64(out), o_ref, what="scale 0.3")


def test_rejects_bad_arguments(fa):
    torch = torch_mod()
    q = torch.zeros((1, 8, 2, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(q, q, q)
    assert e.value.status == -2
    q = torch.zeros((1, 8, 3, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(q, k, k)
    assert e.value.status == -1


def test_binding_checks_caller_buffers(fa):
    """Buffers the caller supplies are checked before any launch: the kernels
    write exactly the sizes they are given, so a short output, a wrong dtype
    or a workspace that is not bytes must never reach them."""
    torch = torch_mod()
    q = torch.zeros((1, 130, 2, 64), dtype=torch.bfloat16, device="cuda")
    bad_outputs = [
        dict(out=torch.empty((1, 129, 2, 64), dtype=torch.bfloat16, device="cuda")),
        dict(out=torch.empty((1, 130, 2, 64), dtype=torch.float16, device="cuda")),
        dict(out=torch.empty((1, 130, 2, 128), dtype=torch.bfloat16, device="cuda")[..., :64]),
        dict(lse=torch.empty((1, 2, 129), dtype=torch.float32, device="cuda")),
        dict(lse=torch.empty((1, 2, 130), dtype=torch.bfloat16, device="cuda")),
        dict(out=torch.empty((1, 130, 2, 64), dtype=torch.bfloat16)),   # host memory
    ]
    for kw in bad_outputs:
        with pytest.raises(ValueError):
            fa.fa_fwd(q, q, q, causal=True, **kw)
        with pytest.raises(ValueError):
            fa.fa_fwd_splitkv(q, q, q, causal=True, **kw)
    with pytest.raises(ValueError):   # a workspace given as fp32 words, not bytes
        fa.fa_fwd_splitkv(q, q, q, workspace=torch.empty(1 << 20, dtype=torch.float32,
                                                         device="cuda"))
    lse = torch.zeros((1, 2, 130), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_bwd(q, q, q, q, lse, q, dq=torch.empty((1, 130, 2, 32), dtype=torch.bfloat16,
                                                      device="cuda"))
    with pytest.raises(ValueError):
        fa.fa_bwd(q, q, q, q, lse[:, :1], q)
    with pytest.raises(ValueError):   # k and v of different shapes
        fa.fa_fwd_varlen(q[0], q[0], q[0, :, :1].contiguous(),
                         torch.tensor([0, 130], dtype=torch.int32, device="cuda"), 130)
    with pytest.raises(ValueError):   # offsets on the host
        fa.fa_fwd_varlen(q[0], q[0], q[0], torch.tensor([0, 130], dtype=torch.int32), 130)
    assert_device_clean()


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_quarter_million_token_sequence_sampled(fa, d, causal):
    """One head over 262,144 tokens (2048 key tiles, 1024 query-tile pairs,
    the last rows seeing every key): the longest sequence of the suite.  The
    oracle evaluates seeded rows plus the first, the middle and the last
    rows, each over all of its visible keys."""
    torch = torch_mod()
    N = 262144
    inp = W.dense_inputs(1, N, 1, 1, d, seed=90 + d)
    out, lse = run_dense(fa, inp, causal)
    rows = np.unique(np.concatenate([
        [0, 1, 127, 128, N // 2, N - 129, N - 2, N - 1],
        np.random.default_rng(91).choice(N, 24, replace=False)]))
    o_ref, l_ref = oracle.attention_one(f64(inp.q[0]), f64(inp.k[0]), f64(inp.v[0]),
                                        causal=causal, rows=rows)
    compare(out[0, rows, 0], o_ref[rows, 0], lse[0, 0, rows], l_ref[0, rows],
            f"N=262144 d{d} causal={causal}")
    assert np.all(np.isfinite(out))
    del out, lse
    torch.cuda.empty_cache()
    assert_device_clean()
