"""GPU parity of chunked prefill over a paged KV cache (fa_fwd_paged)."""
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


def run(fa, inp, causal, k_pool=None, v_pool=None, table=None):
    torch = torch_mod()
    pl = inp.pool
    out, lse = fa.fa_fwd_paged(
        dev_bf16(inp.q), dev_bf16(pl.k_pool if k_pool is None else k_pool),
        dev_bf16(pl.v_pool if v_pool is None else v_pool),
        dev_i32(pl.block_table if table is None else table), dev_i32(pl.ctx_lens),
        dev_i32(inp.cu_seqlens_q), inp.max_seqlen_q, pl.max_ctx_len, causal=causal)
    torch.cuda.synchronize()
    return host_f64(out), lse.cpu().numpy().astype(np.float64)


def ref(inp, causal, seqs=None, heads=None):
    pl = inp.pool
    return oracle.paged_prefill(f64(inp.q), f64(pl.k_pool), f64(pl.v_pool), pl.block_table,
                                pl.ctx_lens, inp.cu_seqlens_q, pl.block_size, causal=causal,
                                seqs=seqs, heads=heads)


# (ctx, q_len): cached prefixes of several sizes, chunks that are the whole
# sequence, single-token chunks, and chunks longer than the context (their
# first queries see no key)
CASES = [(1, 1), (17, 17), (100, 37), (2048, 300), (5000, 1), (129, 129), (3, 10), (700, 260)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (3, 1)])
def test_paged_prefill_ragged(fa, d, causal, H, Hkv):
    """GQA 8 / 2 pairs two query heads per CTA; 3 / 1 pairs two row tiles."""
    ctx = [c for c, _ in CASES]
    ql = [n for _, n in CASES]
    inp = W.paged_prefill_inputs(ctx, ql, H, Hkv, d, seed=50 + H, extra_blocks=3)
    out, lse = run(fa, inp, causal)
    o_ref, l_ref = ref(inp, causal)
    compare(out, o_ref, lse, l_ref, f"paged prefill d{d} causal={causal}")
    if causal:   # sequence 6: ctx 3 < 10 queries, its first 7 queries see nothing
        a = inp.cu_seqlens_q[6]
        assert np.all(out[a:a + 7] == 0) and np.all(np.isneginf(lse[:, a:a + 7]))
    assert_device_clean()


def test_paged_prefill_stale_slots_never_used(fa):
    ctx = [19, 47, 300]
    inp = W.paged_prefill_inputs(ctx, [5, 47, 200], 8, 2, 128, seed=51)
    out, lse = run(fa, inp, True)
    pl = inp.pool
    nan_bits = np.uint16(0x7FC0)
    kp, vp = pl.k_pool.copy(), pl.v_pool.copy()
    for b, c in enumerate(ctx):
        last = pl.block_table[b, (c - 1) // 16]
        used = c - ((c - 1) // 16) * 16
        kp[last, used:] = nan_bits
        vp[last, used:] = nan_bits
    out2, lse2 = run(fa, inp, True, k_pool=kp, v_pool=vp)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    o_ref, l_ref = ref(inp, True)
    compare(out2, o_ref, lse2, l_ref, "paged prefill stale slots")


def test_paged_prefill_matches_varlen_on_contiguous_pool(fa):
    """A chunk covering the whole sequence over an identity block table is
    the varlen causal prefill of the same tokens."""
    torch = torch_mod()
    lengths = [48, 160, 33]
    H, Hkv, d = 4, 2, 128
    var = W.varlen_inputs(lengths, H, Hkv, d, seed=52)
    nb_per = [(L + 15) // 16 for L in lengths]
    pools_k, pools_v, table = [], [], np.full((3, max(nb_per)), -1, dtype=np.int32)
    nb = 0
    for s, L in enumerate(lengths):
        a = var.cu_seqlens[s]
        pad = nb_per[s] * 16 - L
        ks = np.concatenate([var.k[a:a + L], np.zeros((pad, Hkv, d), np.uint16)])
        vs = np.concatenate([var.v[a:a + L], np.zeros((pad, Hkv, d), np.uint16)])
        pools_k.append(ks.reshape(-1, 16, Hkv, d))
        pools_v.append(vs.reshape(-1, 16, Hkv, d))
        table[s, :nb_per[s]] = np.arange(nb, nb + nb_per[s])
        nb += nb_per[s]
    kp = dev_bf16(np.concatenate(pools_k))
    vp = dev_bf16(np.concatenate(pools_v))
    q = dev_bf16(var.q)
    cu = dev_i32(var.cu_seqlens)
    o_p, l_p = fa.fa_fwd_paged(q, kp, vp, dev_i32(table), dev_i32(np.array(lengths)), cu,
                               max(lengths), max(lengths), causal=True)
    o_v, l_v = fa.fa_fwd_varlen(q, dev_bf16(var.k), dev_bf16(var.v), cu, max(lengths),
                                causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_v) and torch.equal(l_p, l_v)


def test_paged_prefill_config_sampled(fa):
    """8 sequences, cached prefixes U[1024, 16384] plus a 1024-token chunk,
    GQA 32/8, d = 128, causal; the oracle checks 2 seeded heads of every
    sequence."""
    cfg = W.WORKLOADS["paged_prefill_gqa_d128"]
    ctx, ql = W.paged_prefill_lengths(cfg["batch"], cfg["prefix_lo"], cfg["prefix_hi"],
                                      cfg["chunk"])
    inp = W.paged_prefill_inputs(ctx, ql, cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    out, lse = run(fa, inp, True)
    heads = sorted(np.random.default_rng(7).choice(cfg["H"], 2, replace=False).tolist())
    o_ref, l_ref = ref(inp, True, heads=heads)
    for h in heads:
        compare(out[:, h], o_ref[:, h], lse[h], l_ref[h], f"paged prefill config head {h}")
    assert np.all(np.isfinite(out))
    assert_device_clean()


def test_paged_prefill_bad_block_flagged(fa):
    inp = W.paged_prefill_inputs([40, 40], [8, 8], 4, 2, 64, seed=53)
    table = inp.pool.block_table.copy()
    table[1, 0] = -5
    fa.fa_device_status(clear=True)
    out, lse = run(fa, inp, True, table=table)
    assert fa.fa_device_status(clear=True) & fa.FA_DEV_BAD_BLOCK
    o_ref, l_ref = ref(inp, True, seqs=[0])
    compare(out[:8], o_ref[:8], lse[:, :8], l_ref[:, :8], "paged prefill unaffected sequence")
