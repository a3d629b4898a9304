"""Failure detection without a GPU fault: a bounded pipeline wait on a
barrier that nothing completes gives up, reports FA_DEV_TIMEOUT through the
status word, and the context keeps working afterwards."""
import time

import numpy as np
import pytest

import oracle
from exact_attention_33_gb300 import workloads as W
from gpu_helpers import compare, dev_bf16, host_f64, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_attention_33_gb300.build import build
    build()
    import exact_attention_33_gb300 as fa_mod
    return fa_mod


def test_bounded_wait_times_out_and_reports(fa):
    torch = torch_mod()
    fa.fa_device_status(clear=True)
    t0 = time.time()
    res = fa.fa_selftest_wait_timeout()
    dt = time.time() - t0
    assert res == 0                     # the wait gave up instead of succeeding
    assert 0.5 < dt < 30.0              # after about the one-second limit
    st = fa.fa_device_status(clear=True)
    assert st & fa.FA_DEV_TIMEOUT
    assert fa.fa_device_status(clear=True) == 0   # cleared
    # the context still runs real work correctly
    inp = W.dense_inputs(1, 130, 2, 2, 64, seed=90)
    out, lse = fa.fa_fwd(dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), causal=True)
    torch.cuda.synchronize()
    f = W.bf16_bits_to_f64
    o_ref, l_ref = oracle.attention_dense(f(inp.q), f(inp.k), f(inp.v), causal=True)
    compare(host_f64(out), o_ref, lse.cpu().numpy(), l_ref, "after timeout self-test")
    assert fa.fa_device_status(clear=True) == 0
