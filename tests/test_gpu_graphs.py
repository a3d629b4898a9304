"""The library's calls inside CUDA graphs.

A serving loop captures a decode step once and replays it: every call here
is asynchronous on the caller's stream, allocates nothing, and launches its
combine as a programmatic dependent of its split grid, which graph capture
keeps as a programmatic edge.  Each test captures a call on fixed device
buffers, writes new inputs into those buffers, replays the graph and
compares the result with the oracle on the new inputs.
"""
import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import assert_device_clean, compare, dev_bf16, dev_i32, host_f64, torch_mod

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


def capture(torch, fn):
    """fn() once eagerly (one-time set-up outside the capture), then captured."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_graph_replay(fa):
    torch = torch_mod()
    ctx = [300, 5000, 17, 2048]
    inp = W.decode_inputs(ctx, 8, 2, 128, seed=60)
    q = dev_bf16(inp.q)
    kp, vp = dev_bf16(inp.k_pool), dev_bf16(inp.v_pool)
    table, cl = dev_i32(inp.block_table), dev_i32(inp.ctx_lens)
    out = torch.empty_like(q)
    lse = torch.empty((len(ctx), 8), dtype=torch.float32, device="cuda")
    ws = fa.new_workspace(fa.fa_decode_workspace_size(len(ctx), 8, 2, 128, inp.max_ctx_len))
    g = capture(torch, lambda: fa.fa_decode_paged(q, kp, vp, table, cl, inp.max_ctx_len,
                                                  out=out, lse=lse, workspace=ws))
    for seed in (61, 62):   # two replays on new queries
        new = W.decode_inputs(ctx, 8, 2, 128, seed=seed)
        q.copy_(dev_bf16(new.q))
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = oracle.paged_decode(f64(new.q), f64(inp.k_pool), f64(inp.v_pool),
                                           inp.block_table, inp.ctx_lens, inp.block_size)
        compare(host_f64(out), o_ref, lse.cpu().numpy().astype(np.float64), l_ref,
                f"decode graph replay seed {seed}")
    assert_device_clean()


@pytest.mark.parametrize("split", [True, False])
def test_prefill_graph_replay(fa, split):
    torch = torch_mod()
    B, N, H, Hkv, d = 1, 1500, 4, 2, 128
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=63)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    if split:
        ws = fa.new_workspace(fa.fa_fwd_splitkv_workspace_size(B, H, N, d, 3))
        fn = lambda: fa.fa_fwd_splitkv(q, k, v, causal=True, num_splits=3, out=out, lse=lse,
                                       workspace=ws)
    else:
        fn = lambda: fa.fa_fwd(q, k, v, causal=True, out=out, lse=lse)
    g = capture(torch, fn)
    new = W.dense_inputs(B, N, H, Hkv, d, seed=64)
    q.copy_(dev_bf16(new.q))
    k.copy_(dev_bf16(new.k))
    v.copy_(dev_bf16(new.v))
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_dense(f64(new.q), f64(new.k), f64(new.v), causal=True)
    compare(host_f64(out), o_ref, lse.cpu().numpy().astype(np.float64), l_ref,
            f"prefill graph replay split={split}")
    assert_device_clean()
