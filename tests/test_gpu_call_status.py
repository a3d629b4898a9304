"""Per-call device status (fa_last_device_status): a data error that only the
device can see is recorded in the workspace of the call that met it, so a
clean call running at the same time on another stream and workspace reports
nothing, and the next call on the same workspace starts from a clean word.
The per-device sticky word (fa_device_status) still gathers every call."""
import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import compare, dev_bf16, dev_i32, host_f64, torch_mod

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


class DecodeCase:
    """Device copies of one seeded decode workload and its output buffers."""

    def __init__(self, ctx, H, Hkv, d, seed, bad_block=None):
        torch = torch_mod()
        self.inp = W.decode_inputs(ctx, H, Hkv, d, seed=seed)
        table = self.inp.block_table.copy()
        if bad_block is not None:
            table[bad_block] = self.inp.num_blocks   # one id past the pool
        self.q = dev_bf16(self.inp.q)
        self.kp, self.vp = dev_bf16(self.inp.k_pool), dev_bf16(self.inp.v_pool)
        self.table, self.ctx = dev_i32(table), dev_i32(self.inp.ctx_lens)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device="cuda")

    def need(self, fa):
        b, H, d = self.q.shape
        return fa.fa_decode_workspace_size(b, H, self.kp.shape[2], d, self.inp.max_ctx_len)

    def run(self, fa, ws):
        fa.fa_decode_paged(self.q, self.kp, self.vp, self.table, self.ctx, self.inp.max_ctx_len,
                           out=self.out, lse=self.lse, workspace=ws)

    def check(self, what):
        o_ref, l_ref = oracle.paged_decode(f64(self.inp.q), f64(self.inp.k_pool),
                                           f64(self.inp.v_pool), self.inp.block_table,
                                           self.inp.ctx_lens, self.inp.block_size)
        compare(host_f64(self.out), o_ref, self.lse.cpu().numpy().astype(np.float64), l_ref,
                what)


def test_bad_block_is_reported_on_its_own_workspace_only(fa):
    torch = torch_mod()
    bad = DecodeCase([3000, 40, 900], 8, 2, 128, seed=70, bad_block=(1, 1))
    clean = DecodeCase([5000, 17, 2048, 700], 8, 2, 128, seed=71)
    ws_bad = fa.new_workspace(max(bad.need(fa), clean.need(fa)))
    ws_clean = fa.new_workspace(clean.need(fa))
    s_bad, s_clean = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    fa.fa_device_status(clear=True)
    with torch.cuda.stream(s_bad):
        bad.run(fa, ws_bad)
    with torch.cuda.stream(s_clean):
        clean.run(fa, ws_clean)
    s_bad.synchronize()
    s_clean.synchronize()
    assert fa.fa_last_device_status(ws_bad) == fa.FA_DEV_BAD_BLOCK
    assert fa.fa_last_device_status(ws_clean) == 0
    clean.check("clean decode beside a failing one")
    # the per-device word gathers every call
    assert fa.fa_device_status(clear=True) == fa.FA_DEV_BAD_BLOCK
    # the word reports the last call: a clean call on the same workspace clears it
    clean.run(fa, ws_bad)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status(ws_bad) == 0
    clean.check("clean decode on the workspace of the failed call")
    assert fa.fa_device_status(clear=True) == 0


def control_block(ws):
    """(acc, last) of a workspace's control block."""
    torch = torch_mod()
    return tuple(int(x) for x in ws[:8].view(torch.int32).cpu())


def test_calls_leave_the_control_block_ready(fa):
    torch = torch_mod()
    bad = DecodeCase([700, 2000], 4, 1, 64, seed=72, bad_block=(0, 3))
    ws = fa.new_workspace(bad.need(fa))
    for _ in range(2):   # the error is reported again by the second call
        bad.run(fa, ws)
        torch.cuda.synchronize()
        assert control_block(ws) == (0, fa.FA_DEV_BAD_BLOCK)
    assert fa.fa_device_status(clear=True) == fa.FA_DEV_BAD_BLOCK


@pytest.mark.parametrize("num_splits", [1, 3])
def test_splitkv_call_status(fa, num_splits):
    """Split-KV prefill publishes its (clean) status both with a combine
    (3 splits) and when one split runs the plain kernel alone."""
    torch = torch_mod()
    B, N, H, Hkv, d = 1, 700, 2, 2, 64
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=73)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    ws = fa.new_workspace(fa.fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits))
    ws[4:8].fill_(0x55)   # a stale `last` word from an earlier call
    for _ in range(2):
        out, lse = fa.fa_fwd_splitkv(q, k, v, causal=True, num_splits=num_splits, workspace=ws)
        torch.cuda.synchronize()
        assert control_block(ws) == (0, 0)
        assert fa.fa_last_device_status(ws) == 0
    o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), causal=True)
    compare(host_f64(out), o_ref, lse.cpu().numpy().astype(np.float64), l_ref,
            f"split-KV prefill, {num_splits} splits")
    assert fa.fa_device_status(clear=True) == 0
