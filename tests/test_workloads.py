"""CPU checks of the seeded input generators (shared by the GPU path and the
oracle): determinism, bf16 rounding, layouts and work counters."""
import numpy as np
import pytest

from exact_attention_33_gb300 import workloads as W


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 100
    x[:4] = [0.0, -0.0, 1.0, -3.5]
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_generator_is_deterministic_and_chunk_stable(monkeypatch):
    a = W.normal_bf16_bits((3, 1000, 7), seed=9, stream=1)
    b = W.normal_bf16_bits((3, 1000, 7), seed=9, stream=1)
    assert np.array_equal(a, b)
    monkeypatch.setattr(W, "_threads", lambda: 1)
    monkeypatch.setattr(W, "CHUNK", 1000)
    c1 = W.normal_bf16_bits((5000,), seed=9, stream=2)
    monkeypatch.setattr(W, "_threads", lambda: 4)
    c4 = W.normal_bf16_bits((5000,), seed=9, stream=2)
    assert np.array_equal(c1, c4)
    assert not np.array_equal(W.normal_bf16_bits((100,), 9, 0), W.normal_bf16_bits((100,), 9, 1))
    x = W.bf16_bits_to_f32(W.normal_bf16_bits((200000,), 1, 0))
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02


def test_outliers_are_exact_powers_of_two():
    inp = W.dense_inputs(1, 300, 2, 2, 64, seed=0, outlier_frac=0.01, outlier_scale=8.0)
    base = W.dense_inputs(1, 300, 2, 2, 64, seed=0)
    for (b, g), rows in inp.outlier_rows.items():
        assert len(rows) == 3
        np.testing.assert_array_equal(W.bf16_bits_to_f32(inp.k[b, rows, g]),
                                      8 * W.bf16_bits_to_f32(base.k[b, rows, g]))
        other = np.setdiff1d(np.arange(300), rows)
        assert np.array_equal(inp.k[b, other, g], base.k[b, other, g])


def test_varlen_and_decode_recipes():
    lengths = W.varlen_lengths()
    assert len(lengths) == 32 and lengths.min() >= 64 and lengths.max() <= 4096
    cu = W.cu_seqlens_from(lengths)
    assert cu[0] == 0 and cu[-1] == lengths.sum() and cu.dtype == np.int32
    ctx = W.decode_ctx_lens()
    assert len(ctx) == 64 and ctx.min() >= 512 and ctx.max() <= 32768
    table, nb = W.paged_block_table(ctx[:5], 16, seed=4)
    used = table[table >= 0]
    assert nb == int(((ctx[:5] + 15) // 16).sum())
    assert np.array_equal(np.sort(used), np.arange(nb))   # a permutation of the pool


def test_counters():
    assert W.prefill_flops(2, 8192, 32, 128, True) == pytest.approx(1.0995e12, rel=1e-4)
    assert W.prefill_flops(4, 2048, 16, 64, False) == pytest.approx(68.7e9, rel=1e-3)
    assert W.varlen_flops([10, 20], 2, 64, False) == 4.0 * (100 + 400) * 64 * 2
    ctx = np.array([16, 17])
    assert W.decode_bytes(ctx, 4, 2, 128, 2) == 33 * 2 * 128 * 4 + 2 * 4 * 128 * 4 + 2 * 4 * 4 + 8 + 3 * 4


def test_e4m3_table_matches_format():
    """OCP E4M3: 1.0 is 0x38, the largest finite value 448 (0x7e), the
    smallest subnormal 2^-9 (0x01), 0x7f / 0xff NaN, sign in bit 7."""
    t = W.e4m3_values()
    assert t[0x38] == 1.0 and t[0xB8] == -1.0
    assert t[0x7e] == 448.0 and np.nanmax(t) == 448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6
    assert np.isnan(t[0x7f]) and np.isnan(t[0xff])
    assert np.all(np.diff(t[:0x7f]) > 0)
    assert np.array_equal(t[0x80:0xff], -t[:0x7f])


def test_e4m3_encode_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100000) * np.exp2(rng.uniform(-12, 8.7, 100000))
    x = x[np.abs(x) <= 448.0].astype(np.float32)   # torch does not saturate
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(W.e4m3_encode(x), ref)
    # ties go to the even code: 1 + 1/16 lies halfway between 1 and 1.125
    assert W.e4m3_encode(np.array([1.0625, 1.1875]))[0] == 0x38
    assert W.e4m3_encode(np.array([1.1875]))[0] == 0x3A
    assert W.e4m3_encode(np.array([1e6, -1e6])).tolist() == [0x7e, 0xfe]


def test_fp8_exact_inputs_give_integer_scores():
    inp = W.fp8_exact_p_inputs(1, 64, 2, 1, 128, seed=1)
    q, k = inp.real("q")[0], inp.real("k")[0]
    s2 = np.einsum("nhd,mhd->hnm", q, np.repeat(k, 2, axis=1)) * inp.scale / np.log(2.0)
    assert np.allclose(s2, np.round(s2), atol=1e-12) and np.abs(s2).max() <= 4
    assert inp.v_descale == 0.25 and np.all(np.abs(W.e4m3_decode(inp.v)) <= 8)
