"""GPU parity of paged GQA flash-decoding (fa_decode_paged)."""
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


def run_decode(fa, inp, k_pool=None, v_pool=None, table=None):
    torch = torch_mod()
    out, lse = fa.fa_decode_paged(
        dev_bf16(inp.q), dev_bf16(inp.k_pool if k_pool is None else k_pool),
        dev_bf16(inp.v_pool if v_pool is None else v_pool),
        dev_i32(inp.block_table if table is None else table), dev_i32(inp.ctx_lens),
        inp.max_ctx_len)
    torch.cuda.synchronize()
    return host_f64(out), lse.cpu().numpy().astype(np.float64)


def ref_decode(inp, batches=None, heads=None):
    return oracle.paged_decode(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool), inp.block_table,
                               inp.ctx_lens, inp.block_size, batches=batches, heads=heads)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_ragged_contexts(fa, d):
    ctx = [1, 15, 16, 17, 100, 513, 2048, 0, 4099]
    inp = W.decode_inputs(ctx, 8, 2, d, seed=40, extra_blocks=5)
    out, lse = run_decode(fa, inp)
    o_ref, l_ref = ref_decode(inp)
    compare(out, o_ref, lse, l_ref, f"decode d{d}")
    assert np.all(out[7] == 0) and np.all(np.isneginf(lse[7]))
    assert_device_clean()


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
def test_decode_gqa_groups(fa, group):
    ctx = [33, 700, 1500]
    inp = W.decode_inputs(ctx, 2 * group, 2, 128, seed=41 + group)
    out, lse = run_decode(fa, inp)
    o_ref, l_ref = ref_decode(inp)
    compare(out, o_ref, lse, l_ref, f"decode group {group}")


def test_decode_stale_slots_never_used(fa):
    """Slots of the last block past ctx_len hold NaN: the result must not change."""
    ctx = [3, 18, 31, 47]
    inp = W.decode_inputs(ctx, 8, 2, 128, seed=42)
    out, lse = run_decode(fa, inp)
    nan_bits = np.uint16(0x7FC0)
    kp, vp = inp.k_pool.copy(), inp.v_pool.copy()
    for b, c in enumerate(ctx):
        last = inp.block_table[b, (c - 1) // 16]
        used = c - ((c - 1) // 16) * 16
        kp[last, used:] = nan_bits
        vp[last, used:] = nan_bits
    out2, lse2 = run_decode(fa, inp, k_pool=kp, v_pool=vp)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    o_ref, l_ref = ref_decode(inp)
    compare(out2, o_ref, lse2, l_ref, "decode stale slots")


def test_decode_config_full(fa):
    """Full-size step: batch 64, 32 query / 8 KV heads, d 128, ctx U[512, 32768],
    16-token blocks in a randomly permuted pool; every (batch, head) checked."""
    cfg = W.WORKLOADS["paged_decode_gqa_d128"]
    ctx = W.decode_ctx_lens(cfg["batch"], cfg["ctx_lo"], cfg["ctx_hi"])
    inp = W.decode_inputs(ctx, cfg["H"], cfg["Hkv"], cfg["d"], cfg["block_size"], seed=0)
    out, lse = run_decode(fa, inp)
    o_ref, l_ref = ref_decode(inp)
    compare(out, o_ref, lse, l_ref, "decode config")
    assert_device_clean()


def test_decode_bad_block_id_is_flagged(fa):
    torch = torch_mod()
    ctx = [40, 40]
    inp = W.decode_inputs(ctx, 4, 2, 128, seed=43)
    table = inp.block_table.copy()
    table[1, 1] = inp.num_blocks          # out of range
    fa.fa_device_status(clear=True)
    out, lse = run_decode(fa, inp, table=table)
    assert fa.fa_device_status(clear=True) & fa.FA_DEV_BAD_BLOCK
    o_ref, l_ref = ref_decode(inp, batches=[0])
    compare(out[0], o_ref[0], lse[0], l_ref[0], "decode row unaffected by the bad row")


def test_decode_workspace_too_small(fa):
    torch = torch_mod()
    inp = W.decode_inputs([100], 4, 2, 64, seed=44)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_decode_paged(dev_bf16(inp.q), dev_bf16(inp.k_pool), dev_bf16(inp.v_pool),
                           dev_i32(inp.block_table), dev_i32(inp.ctx_lens), inp.max_ctx_len,
                           workspace=ws)
    assert e.value.status == -4


def test_decode_binding_checks_caller_buffers(fa):
    """The decode calls check the pools, the table, the context lengths and
    the caller's outputs before any launch (the no-allocation call included:
    its output is always the caller's)."""
    torch = torch_mod()
    inp = W.decode_inputs([40, 70], 4, 2, 128, seed=44)
    q, kp, vp = dev_bf16(inp.q), dev_bf16(inp.k_pool), dev_bf16(inp.v_pool)
    table, ctx = dev_i32(inp.block_table), dev_i32(inp.ctx_lens)
    good_out = torch.empty_like(q)
    with pytest.raises(ValueError):   # v_pool shape differs from k_pool
        fa.fa_decode_paged(q, kp, vp[:-1].contiguous(), table, ctx, inp.max_ctx_len)
    with pytest.raises(ValueError):   # one context length too few
        fa.fa_decode_paged(q, kp, vp, table, ctx[:1].contiguous(), inp.max_ctx_len)
    with pytest.raises(ValueError):   # table rows do not match the batch
        fa.fa_decode_paged(q, kp, vp, table[:1].contiguous(), ctx, inp.max_ctx_len)
    with pytest.raises(ValueError):
        fa.fa_decode_paged(q, kp, vp, table, ctx, inp.max_ctx_len,
                           out=torch.empty((2, 4, 64), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.fa_decode_paged_noalloc(q, kp, vp, table, ctx, inp.max_ctx_len,
                                   out=good_out[:1].contiguous())
    with pytest.raises(ValueError):
        fa.fa_decode_paged_noalloc(q, kp, vp, table, ctx, inp.max_ctx_len, out=good_out,
                                   lse=torch.empty((2, 4), dtype=torch.float64, device="cuda"))
    out, lse = fa.fa_decode_paged_noalloc(q, kp, vp, table, ctx, inp.max_ctx_len, out=good_out,
                                          lse=torch.empty((2, 4), dtype=torch.float32,
                                                          device="cuda"))
    torch.cuda.synchronize()
    o_ref, l_ref = ref_decode(inp)
    compare(host_f64(out), o_ref, lse.cpu().numpy().astype(np.float64), l_ref, "noalloc binding")
    assert_device_clean()


def test_decode_quarter_million_token_context(fa):
    """Contexts of 262,144 tokens (16,384 blocks, 512 key splits, all merged
    by one combine row) beside single-token, odd-length and empty contexts,
    on a pool of about 20,000 blocks in random order."""
    ctx = [262144, 1, 70001, 0]
    inp = W.decode_inputs(ctx, 8, 2, 128, seed=45, extra_blocks=7)
    out, lse = run_decode(fa, inp)
    o_ref, l_ref = ref_decode(inp)
    compare(out, o_ref, lse, l_ref, "decode 262144-token context")
    assert_device_clean()


@pytest.mark.parametrize("ctx", [[5, 40, 17, 1, 90], [700, 3, 1200]])
def test_decode_combine_row_layouts(fa, ctx):
    """Odd numbers of (sequence, head) rows (5 x 3 and 3 x 3 heads): short
    contexts merge one row per warp, four rows per CTA, so the last CTA holds
    rows past the end; longer ones merge each row with four warps."""
    inp = W.decode_inputs(ctx, 3, 1, 128, seed=46 + len(ctx))
    out, lse = run_decode(fa, inp)
    o_ref, l_ref = ref_decode(inp)
    compare(out, o_ref, lse, l_ref, f"decode rows {len(ctx)} x 3")
    assert_device_clean()
