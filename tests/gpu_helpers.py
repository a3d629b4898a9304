"""Helpers shared by the GPU parity tests: move seeded bf16 inputs to the
device, run the CUDA path through the C ABI binding, and compare with the
fp64 oracle at the stated tolerance.

Tolerance (bf16 inputs, fp32 accumulation, bf16 output):
  max |out - oracle| <= 2e-2, mean |out - oracle| <= 2e-3,
  |lse - oracle_lse| <= 1e-3 (and both -inf together).
"""

from __future__ import annotations

import numpy as np

TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE = 1e-3


def torch_mod():
    import torch
    return torch


def dev_bf16(bits: np.ndarray):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev_i32(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def compare(out, out_ref, lse=None, lse_ref=None, what="", mask=None):
    """Element-wise comparison; ``mask`` selects the entries to compare."""
    out = np.asarray(out, dtype=np.float64)
    out_ref = np.asarray(out_ref, dtype=np.float64)
    if mask is not None:
        out, out_ref = out[mask], out_ref[mask]
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - out_ref)
    mx = float(err.max()) if err.size else 0.0
    mean = float(err.mean()) if err.size else 0.0
    assert mx <= TOL_MAX, f"{what}: max |err| {mx:.3e} > {TOL_MAX}"
    assert mean <= TOL_MEAN, f"{what}: mean |err| {mean:.3e} > {TOL_MEAN}"
    res = {"max_err": mx, "mean_err": mean}
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        if mask is not None and mask.shape == lse.shape:
            lse, lse_ref = lse[mask], lse_ref[mask]
        fin = np.isfinite(lse_ref)
        assert np.array_equal(fin, np.isfinite(lse)), f"{what}: lse finiteness differs"
        lerr = float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
        assert lerr <= TOL_LSE, f"{what}: max |lse err| {lerr:.3e} > {TOL_LSE}"
        res["lse_err"] = lerr
    return res


def assert_device_clean():
    import exact_attention_33_gb300 as fa
    st = fa.fa_device_status(clear=True)
    assert st == 0, f"device status word set: {st:#x}"
