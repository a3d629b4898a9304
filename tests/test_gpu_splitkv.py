"""GPU parity of the split-KV dense prefill (fa_fwd_splitkv)."""
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


def f64(bits):
    return W.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(1, 0), (200, 2), (1000, 3), (1000, 7), (3000, 0),
                                      (3000, 16), (2500, 1)])
def test_splitkv_small(fa, d, causal, N, splits):
    torch = torch_mod()
    inp = W.dense_inputs(1, N, 2, 1, d, seed=70 + N)
    out, lse = fa.fa_fwd_splitkv(dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v),
                                 causal=causal, num_splits=splits)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), causal=causal)
    compare(host_f64(out), o_ref, lse.cpu().numpy(), l_ref,
            f"splitkv N{N} d{d} causal={causal} splits={splits}")
    assert_device_clean()


def test_splitkv_single_long_sequence_sampled(fa):
    """B = 1, 4 heads, N = 16384, d = 128, causal, library-chosen splits;
    the oracle evaluates 256 seeded rows of every head."""
    torch = torch_mod()
    inp = W.dense_inputs(1, 16384, 4, 4, 128, seed=0)
    out, lse = fa.fa_fwd_splitkv(dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), causal=True)
    torch.cuda.synchronize()
    out = host_f64(out)
    lse = lse.cpu().numpy()
    rows = np.sort(np.random.default_rng(8).choice(16384, 256, replace=False))
    o_ref, l_ref = oracle.attention_one(f64(inp.q[0]), f64(inp.k[0]), f64(inp.v[0]), causal=True,
                                        rows=rows)
    compare(out[0][rows], o_ref[rows], lse[0][:, rows], l_ref[:, rows], "splitkv long sampled")
    assert np.all(np.isfinite(out))
    assert_device_clean()


def test_splitkv_workspace_checks(fa):
    torch = torch_mod()
    inp = W.dense_inputs(1, 300, 2, 2, 64, seed=71)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    need = fa.fa_fwd_splitkv_workspace_size(1, 2, 300, 64, 3)
    assert need >= 3 * 300 * 2 * 64 * 4
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv(q, k, v, num_splits=3, workspace=ws)
    assert e.value.status == -4


def test_splitkv_bench_workload_full(fa):
    """The split-KV leg's workload (B=1, H=4, N=8192, d=128, causal, splits
    chosen by the library), every element compared."""
    torch = torch_mod()
    cfg = W.WORKLOADS["splitkv_small_bh_d128"]
    inp = W.dense_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    out, lse = fa.fa_fwd_splitkv(dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), causal=True)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_dense(f64(inp.q), f64(inp.k), f64(inp.v), causal=True)
    compare(host_f64(out), o_ref, lse.cpu().numpy(), l_ref, "splitkv bench workload")
    assert_device_clean()
