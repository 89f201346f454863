"""Pins for the flat-GEMM oracle (CPU only).

The oracle is ``Y = X W^T`` for the decode-phase projections of
"【FlashAttention-V4，非官方】FlashDecoding++" (sections 1, 2 and 4). None of these
re-types that product: each pin checks an identity or permutation weight matrix, a
hand-derived fixture, a brute-force ``math.fsum`` loop, linearity, the GEMV special
case, or the page's zero padding of the token dimension. ``test_planted_*`` checks that
plausible slips (a transposed operand, a dropped or shifted K column, a sign flip, the
wrong output orientation) each fail at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_derived.json")
rng = np.random.default_rng(2024)


def check_identity(f):
    x = rng.normal(size=(5, 7))
    return np.array_equal(f(x, np.eye(7)), x)


def check_permutation(f):
    # w[n, k] = 1 iff k = perm[n], so y[m, n] = x[m, perm[n]]; a 3-cycle is not its own inverse
    K = 6
    perm = np.array([1, 2, 0, 4, 5, 3])
    w = np.zeros((K, K))
    w[np.arange(K), perm] = 1.0
    x = rng.normal(size=(3, K))
    return np.array_equal(f(x, w), x[:, perm])


def check_selector_rows(f):
    # a non-square weight: N = 2 outputs picking column 4 and summing columns 0 and 2
    x = rng.normal(size=(4, 5))
    w = np.array([[0, 0, 0, 0, 1.0], [1.0, 0, 1.0, 0, 0]])
    y = f(x, w)
    return y.shape == (4, 2) and np.allclose(y[:, 0], x[:, 4], atol=0) and np.allclose(
        y[:, 1], x[:, 0] + x[:, 2], atol=1e-15)


def check_brute_force(f):
    for M, K, N in [(1, 1, 1), (1, 9, 4), (3, 5, 2), (8, 16, 3), (2, 33, 7)]:
        x = rng.normal(size=(M, K))
        w = rng.normal(size=(N, K))
        y = f(x, w)
        if y.shape != (M, N):
            return False
        for m in range(M):
            for n in range(N):
                if abs(y[m, n] - math.fsum(x[m, k] * w[n, k] for k in range(K))) > 1e-12:
                    return False
    return True


def check_linearity(f):
    x1, x2 = rng.normal(size=(4, 12)), rng.normal(size=(4, 12))
    w1, w2 = rng.normal(size=(6, 12)), rng.normal(size=(6, 12))
    a, b = 0.75, -2.5
    ok = np.allclose(f(a * x1 + b * x2, w1), a * f(x1, w1) + b * f(x2, w1), atol=1e-12)
    return ok and np.allclose(f(x1, a * w1 + b * w2), a * f(x1, w1) + b * f(x1, w2), atol=1e-12)


def check_gemv(f):
    # one token: y is the combination of W's columns weighted by x
    K, N = 10, 6
    x = rng.normal(size=(1, K))
    w = rng.normal(size=(N, K))
    want = np.zeros(N)
    for k in range(K):
        want = want + x[0, k] * w[:, k]
    return np.allclose(f(x, w)[0], want, atol=1e-13)


def check_zero_padding(f):
    # the page pads the token dimension with zero rows (to 8; libraries to 64): the real
    # rows keep their values and the padded rows are zero
    x = rng.normal(size=(3, 20))
    w = rng.normal(size=(9, 20))
    y = f(x, w)
    for mult in (8, 64):
        xp = oracle.pad_rows(x, mult)
        if xp.shape != (mult, 20) or np.any(xp[3:] != 0) or np.any(xp[:3] != x):
            return False
        yp = f(xp, w)
        if not (np.allclose(yp[:3], y, atol=0) and np.all(yp[3:] == 0)):
            return False
    return True


def check_golden(f):
    with open(GOLDEN) as fh:
        cases = [c for c in json.load(fh)["cases"] if c["kind"] == "flat_gemm"]
    assert cases
    return all(np.allclose(f(np.array(c["x"]), np.array(c["w"])), c["y"], atol=1e-14) for c in cases)


PINS = [check_identity, check_permutation, check_selector_rows, check_brute_force, check_linearity,
        check_gemv, check_zero_padding, check_golden]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_flat_gemm_pins(pin):
    assert pin(oracle.flat_gemm)


def test_flat_gemm_rejects_mismatched_k():
    with pytest.raises(ValueError):
        oracle.flat_gemm(np.zeros((2, 3)), np.zeros((4, 5)))


def _mutant(kind):
    def f(x, w):
        x = np.asarray(x, float)
        w = np.asarray(w, float)
        if kind == "transposed_w":          # X W instead of X W^T (square shapes only)
            return x @ w if x.shape[1] == w.shape[0] else x @ w.T * 0 + np.nan
        if kind == "drop_last_k":
            return x[:, :-1] @ w[:, :-1].T
        if kind == "shift_k":
            return x @ np.roll(w, 1, axis=1).T
        if kind == "sign":
            return -(x @ w.T)
        if kind == "output_transposed":     # W X^T instead of X W^T
            return (x @ w.T).T
        if kind == "fp32_accumulate":       # accumulating in fp32 misses the fp64 bar
            return (x.astype(np.float32) @ w.T.astype(np.float32)).astype(np.float64)
        raise ValueError(kind)
    return f


@pytest.mark.parametrize("kind", ["transposed_w", "drop_last_k", "shift_k", "sign", "output_transposed",
                                  "fp32_accumulate"])
def test_planted_flat_gemm_mistakes_are_caught(kind):
    mutant = _mutant(kind)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin(mutant)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"mutant {kind} passed every pin"
