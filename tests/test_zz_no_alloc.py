"""GPU test of fa_decode_paged_noalloc, the paged decode that allocates
nothing: its split partial states live in the library's static device
scratch array instead of a caller workspace.  It serves callers that cannot
call cudaMalloc (a plugin whose host framework owns all device memory, or a
decode loop that must avoid cudaMalloc/cudaFree and their implicit device
synchronisation).

The entry point is called through the C ABI on two calls in a row (different
inputs, the second needing fewer splits than the first, so stale scratch
from the first call would show) and each result is checked against the
workspace-taking fa_decode_paged on the same inputs, at the tolerance of the
other parity tests.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

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


def _call_noalloc(lib, q, kp, vp, table, ctx, max_ctx, out, lse, scale):
    torch = torch_mod()
    batch, H, d = q.shape
    num_blocks, block_size, Hkv, _ = kp.shape
    P = ctypes.c_void_p
    return lib.fa_decode_paged_noalloc(
        P(q.data_ptr()), P(kp.data_ptr()), P(vp.data_ptr()), P(table.data_ptr()),
        table.shape[1], P(ctx.data_ptr()), max_ctx, batch, H, Hkv, d, block_size, num_blocks,
        ctypes.c_float(scale), P(out.data_ptr()), P(lse.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_decode_twice(fa):
    torch = torch_mod()
    lib = fa.load_library()
    cases = [([3000, 17, 900, 4096, 1, 2500], 32, 8, 128, 60),
             ([40, 700, 16, 5], 16, 4, 64, 61)]
    for ctx, H, Hkv, d, seed in cases:
        inp = W.decode_inputs(ctx, H, Hkv, d, seed=seed)
        q, kp, vp = dev_bf16(inp.q), dev_bf16(inp.k_pool), dev_bf16(inp.v_pool)
        table, ctx_d = dev_i32(inp.block_table), dev_i32(inp.ctx_lens)
        need = fa.fa_decode_workspace_size(len(ctx), H, Hkv, d, inp.max_ctx_len)
        assert 0 < need <= fa.FA_DECODE_NOALLOC_SCRATCH_BYTES
        scale = 1.0 / np.sqrt(d)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        rc = _call_noalloc(lib, q, kp, vp, table, ctx_d, inp.max_ctx_len, out, lse, scale)
        assert rc == 0, fa.fa_status_string(rc)
        ref_out, ref_lse = fa.fa_decode_paged(q, kp, vp, table, ctx_d, inp.max_ctx_len,
                                              scale=scale)
        torch.cuda.synchronize()
        compare(host_f64(out), host_f64(ref_out), lse.cpu().numpy(), ref_lse.cpu().numpy(),
                f"noalloc vs workspace decode {ctx}")
    assert fa.fa_device_status(clear=True) == 0


def test_noalloc_rejects_requests_beyond_the_static_scratch(fa):
    torch = torch_mod()
    lib = fa.load_library()
    batch, H, Hkv, d, max_ctx = 64, 32, 8, 128, 32768
    assert fa.fa_decode_workspace_size(batch, H, Hkv, d, max_ctx) > \
        fa.FA_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((batch, H, d), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((4, 16, Hkv, d), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((batch, max_ctx // 16), dtype=torch.int32, device="cuda")
    ctx = torch.zeros((batch,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((batch, H), dtype=torch.float32, device="cuda")
    rc = _call_noalloc(lib, q, kp, kp, table, ctx, max_ctx, out, lse, 0.1)
    assert rc == -4
