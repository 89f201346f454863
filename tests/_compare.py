"""Tolerance checks shared by the GPU parity tests.

The bars: fp32 inputs, max-abs error <= 1e-4; bf16 inputs with fp32
accumulation, max-abs <= 2e-2 and mean-abs <= 2e-3. Both apply to the output
and to the LSE. Operation order changes float results, so tolerances are set
per dtype ("快速注意力内核与算子融合", notes on verifying compiled results).
"""
import numpy as np

TOL = {"f32": dict(max_abs=1e-4, mean_abs=1e-4), "bf16": dict(max_abs=2e-2, mean_abs=2e-3)}


def assert_close(got, want, dtype_name, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    inf_w = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf_w), f"{what}: infinities differ"
    assert np.array_equal(got[inf_w], want[inf_w]), f"{what}: signs of infinities differ"
    assert not np.isnan(got[~inf_w]).any(), f"{what}: NaN in result"
    err = np.abs(got[~inf_w] - want[~inf_w])
    if err.size == 0:
        return 0.0, 0.0
    tol = TOL[dtype_name]
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= tol["max_abs"], f"{what}: max-abs {mx:.3e} > {tol['max_abs']}"
    assert mean <= tol["mean_abs"], f"{what}: mean-abs {mean:.3e} > {tol['mean_abs']}"
    return mx, mean
