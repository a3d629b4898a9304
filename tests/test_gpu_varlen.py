"""GPU parity of the packed varlen prefill path (fa_fwd_varlen)."""
import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import (assert_device_clean, compare, dev_bf16, dev_i32, host_f64, torch_mod)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_attention_33_gb300.build import build
    build()
    import exact_attention_33_gb300 as fa_mod
    fa_mod.fa_device_status(clear=True)
    return fa_mod


def f64(bits):
    return W.bf16_bits_to_f64(bits)


def run_varlen(fa, inp, causal):
    torch = torch_mod()
    out, lse = fa.fa_fwd_varlen(dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v),
                                dev_i32(inp.cu_seqlens), inp.max_seqlen, causal=causal)
    torch.cuda.synchronize()
    return host_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (8, 2), (3, 1)])
def test_varlen_ragged(fa, d, causal, H, Hkv):
    """Short sequences: an even GQA group pairs two query heads per CTA (H 4
    and 8), an odd one runs one query tile per CTA (H 3 over one KV head)."""
    lengths = [1, 5, 128, 129, 300, 0, 700, 256, 2]
    inp = W.varlen_inputs(lengths, H, Hkv, d, seed=30 + H)
    out, lse = run_varlen(fa, inp, causal)
    o_ref, l_ref = oracle.attention_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens,
                                           causal=causal)
    compare(out, o_ref, lse, l_ref, f"varlen H{H}/{Hkv} d{d} causal={causal}")
    assert_device_clean()


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_varlen_long_sequences(fa, d, causal):
    """Batches of 4096 rows or more per sequence on average run two query
    tiles per CTA (the shorter batches above run one): ragged long sequences
    with GQA, every element against the oracle."""
    lengths = [4100, 5000, 4300]
    inp = W.varlen_inputs(lengths, 2, 1, d, seed=33)
    out, lse = run_varlen(fa, inp, causal)
    o_ref, l_ref = oracle.attention_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens,
                                           causal=causal)
    compare(out, o_ref, lse, l_ref, f"long varlen d{d} causal={causal}")
    assert_device_clean()


@pytest.mark.parametrize("num_seqs", [100, 150])
def test_varlen_many_sequences(fa, num_seqs):
    """More than 32 sequences: the padding-free order looks its item up over
    several 32-sequence chunks (up to 128 sequences); beyond 128 the launch
    uses the padded order, whose CTAs past a sequence's end leave at once.
    Short ragged lengths (zero included), causal, GQA, every element."""
    lengths = np.random.default_rng(34 + num_seqs).integers(0, 300, num_seqs)
    inp = W.varlen_inputs(lengths, 4, 2, 64, seed=35)
    out, lse = run_varlen(fa, inp, True)
    o_ref, l_ref = oracle.attention_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens,
                                           causal=True)
    compare(out, o_ref, lse, l_ref, f"varlen {num_seqs} sequences")
    assert_device_clean()


def test_varlen_config_sampled(fa):
    """Full-size packed batch (32 sequences, lengths U[64, 4096], GQA 16/4,
    d = 128, causal); the oracle evaluates every sequence for 2 seeded heads."""
    cfg = W.WORKLOADS["varlen_gqa_d128"]
    lengths = W.varlen_lengths(cfg["num_seqs"], cfg["len_lo"], cfg["len_hi"])
    inp = W.varlen_inputs(lengths, cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    out, lse = run_varlen(fa, inp, True)
    heads = sorted(np.random.default_rng(6).choice(cfg["H"], 2, replace=False).tolist())
    for h in heads:
        g = h // (cfg["H"] // cfg["Hkv"])
        o_ref, l_ref = oracle.attention_varlen(f64(inp.q[:, h:h + 1]), f64(inp.k[:, g:g + 1]),
                                               f64(inp.v[:, g:g + 1]), inp.cu_seqlens,
                                               causal=True)
        compare(out[:, h], o_ref[:, 0], lse[h], l_ref[0], f"varlen config head {h}")
    assert np.all(np.isfinite(out))
    assert_device_clean()


def test_varlen_equal_lengths_match_dense(fa):
    """Equal-length packing is the dense layout: both paths give the same bits."""
    torch = torch_mod()
    B, N, H, Hkv, d = 3, 333, 4, 2, 128
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=31)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    o_d, l_d = fa.fa_fwd(q, k, v, causal=True)
    cu = dev_i32(np.arange(B + 1) * N)
    o_v, l_v = fa.fa_fwd_varlen(q.view(B * N, H, d), k.view(B * N, Hkv, d),
                                v.view(B * N, Hkv, d), cu, N, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_d.view(B * N, H, d), o_v)
    assert torch.equal(l_d.permute(1, 0, 2).reshape(H, B * N), l_v)


def test_varlen_bad_cu_seqlens_flagged(fa):
    torch = torch_mod()
    inp = W.varlen_inputs([10, 20], 2, 2, 64, seed=32)
    bad = np.array([0, 25, 20], dtype=np.int32)   # decreasing: sequence 1 is invalid
    fa.fa_device_status(clear=True)
    fa.fa_fwd_varlen(dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_i32(bad), 25)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) & fa.FA_DEV_BAD_SEQLEN


@pytest.mark.parametrize("H,Hkv", [(4, 2), (3, 1)])
def test_varlen_max_seqlen_too_small_is_flagged(fa, H, Hkv):
    """A sequence longer than the max_seqlen the caller states (200 rows
    against 100) cannot be covered by a grid sized from it: the call sets
    FA_DEV_BAD_SEQLEN, with head pairs (H 4 / 2) and one tile per CTA (3 / 1)
    alike.  The same batch with the true maximum matches the oracle."""
    torch = torch_mod()
    inp = W.varlen_inputs([100, 200], H, Hkv, 64, seed=36 + H)
    q, k, v, cu = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_i32(inp.cu_seqlens)
    fa.fa_device_status(clear=True)
    fa.fa_fwd_varlen(q, k, v, cu, 100, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) & fa.FA_DEV_BAD_SEQLEN
    out, lse = fa.fa_fwd_varlen(q, k, v, cu, 200, causal=True)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens,
                                           causal=True)
    compare(host_f64(out), o_ref, lse.cpu().numpy().astype(np.float64), l_ref,
            f"varlen H{H}/{Hkv} true max_seqlen")
    assert_device_clean()
