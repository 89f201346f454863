"""Pins for the fp64 oracle, checked against what the definition fixes (CPU only).

None of these re-types the oracle's own formula. Each one checks a closed form, a
special case, an invariant, a hand-derived fixture or a brute-force loop. Every
pin is chosen so that a plausible slip in the oracle fails at least one of them.
``test_planted_mistakes_are_caught`` checks that against deliberately broken copies.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_attention_28_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_derived.json")
rng = np.random.default_rng(12345)


def _arr(x):
    return np.array(x, dtype=object).astype(np.float64) if any(
        isinstance(v, str) for v in np.ravel(np.array(x, dtype=object))) else np.array(x, float)


# ----------------------------------------------------------------------------- attend

def check_single_key(attend):
    q = rng.normal(size=(3, 8))
    k = rng.normal(size=(1, 8))
    v = rng.normal(size=(1, 8))
    out, lse = attend(q, k, v, 0.3)
    ok = np.allclose(out, np.repeat(v, 3, axis=0), atol=1e-14)
    expect_lse = [0.3 * math.fsum(q[i, d] * k[0, d] for d in range(8)) for i in range(3)]
    return ok and np.allclose(lse, expect_lse, atol=1e-13)


def check_identical_values(attend):
    q = rng.normal(size=(4, 16))
    k = rng.normal(size=(9, 16)) * 3
    row = rng.normal(size=16)
    v = np.tile(row, (9, 1))
    out, _ = attend(q, k, v, 0.25)
    return np.allclose(out, np.tile(row, (4, 1)), atol=1e-13)


def check_identical_keys(attend):
    q = rng.normal(size=(2, 8))
    kr = rng.normal(size=8)
    k = np.tile(kr, (5, 1))
    v = rng.normal(size=(5, 8))
    out, lse = attend(q, k, v, 0.5)
    s = [0.5 * math.fsum(q[i] * kr) for i in range(2)]
    return (np.allclose(out, np.tile(v.mean(axis=0), (2, 1)), atol=1e-13)
            and np.allclose(lse, [x + math.log(5) for x in s], atol=1e-13))


def check_two_key_closed_form(attend):
    q = rng.normal(size=(1, 4))
    k = rng.normal(size=(2, 4))
    v = rng.normal(size=(2, 4))
    scale = 0.7
    s1 = scale * math.fsum(q[0] * k[0])
    s2 = scale * math.fsum(q[0] * k[1])
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))                  # logistic weight of key 1
    out, lse = attend(q, k, v, scale)
    return (np.allclose(out[0], w1 * v[0] + (1 - w1) * v[1], atol=1e-13)
            and abs(lse[0] - (s1 + math.log1p(math.exp(s2 - s1)))) < 1e-13)


def check_brute_force(attend):
    """Pure-Python loops, no max subtraction (logits kept small), fsum everywhere."""
    n, L, D = 3, 7, 5
    q = rng.normal(size=(n, D))
    k = rng.normal(size=(L, D))
    v = rng.normal(size=(L, D))
    scale = 0.45
    out, lse = attend(q, k, v, scale)
    for i in range(n):
        e = [math.exp(scale * math.fsum(q[i][d] * k[j][d] for d in range(D))) for j in range(L)]
        z = math.fsum(e)
        for d in range(D):
            ref = math.fsum(e[j] * v[j][d] for j in range(L)) / z
            if abs(out[i, d] - ref) > 1e-13:
                return False
        if abs(lse[i] - math.log(z)) > 1e-13:
            return False
    return True


def check_weights_form_distribution(attend):
    """With V = identity the output row is the weight vector: >= 0, sums to 1, ratios e^(s_i - s_j)."""
    D = 6
    q = rng.normal(size=(2, D))
    k = rng.normal(size=(D, D))
    out, _ = attend(q, k, np.eye(D), 0.9)
    if (out < 0).any() or not np.allclose(out.sum(axis=1), 1.0, atol=1e-12):
        return False
    s = 0.9 * np.array([[math.fsum(q[i] * k[j]) for j in range(D)] for i in range(2)])
    return np.allclose(np.log(out[:, 1:] / out[:, :1]), s[:, 1:] - s[:, :1], atol=1e-12)


def check_shift_invariance_large_logits(attend):
    """Adding a constant c to every logit leaves out unchanged and moves lse by c, even for c = 1000."""
    q = rng.normal(size=(2, 4))
    k = rng.normal(size=(6, 4))
    v = rng.normal(size=(6, 4))
    o1, l1 = attend(q, k, v, 1.0)
    q2 = np.concatenate([q, np.full((2, 1), 1000.0)], axis=1)
    k2 = np.concatenate([k, np.ones((6, 1))], axis=1)
    o2, l2 = attend(q2, k2, v, 1.0)
    return np.isfinite(o2).all() and np.allclose(o1, o2, atol=1e-12) and np.allclose(l2 - l1, 1000.0, atol=1e-9)


def check_dominant_key(attend):
    """Logits spread over 800: the top key takes all the weight (e^-800 is 0 in fp64)."""
    k = np.zeros((5, 2))
    k[:, 0] = [0.0, -1.0, 1.0, -0.5, 0.2]
    k[3, 1] = 1.0
    q = np.array([[0.0, 800.0]])
    v = rng.normal(size=(5, 3))
    out, lse = attend(q, k, v, 1.0)
    return np.isfinite(out).all() and np.allclose(out[0], v[3], atol=1e-14) and abs(lse[0] - 800.0) < 1e-9


def check_empty_keys(attend):
    out, lse = attend(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    return np.all(out == 0) and np.all(lse == -np.inf)


ATTEND_PINS = [check_single_key, check_identical_values, check_identical_keys,
               check_two_key_closed_form, check_brute_force, check_weights_form_distribution,
               check_shift_invariance_large_logits, check_dominant_key, check_empty_keys]


@pytest.mark.parametrize("pin", ATTEND_PINS, ids=lambda f: f.__name__)
def test_attend_pins(pin):
    assert pin(oracle.attend)


# ----------------------------------------------------------------------------- golden

def _golden(kind):
    with open(GOLDEN) as f:
        return [c for c in json.load(f)["cases"] if c["kind"] == kind]


def test_golden_attend():
    for c in _golden("attend"):
        out, lse = oracle.attend(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]), c["scale"])
        np.testing.assert_allclose(out, c["out"], atol=1e-13)
        np.testing.assert_allclose(lse, c["lse"], atol=1e-13)


def test_golden_prefill():
    for c in _golden("prefill"):
        T = len(c["q"])
        q = np.array(c["q"]).reshape(1, T, 1, 1)
        k = np.array(c["k"]).reshape(1, T, 1, 1)
        v = np.array(c["v"]).reshape(1, T, 1, 1)
        out, lse = oracle.prefill_causal(q, k, v, c["scale"])
        np.testing.assert_allclose(out[0, :, 0, 0], c["out"], atol=1e-12)
        np.testing.assert_allclose(lse[0, 0], c["lse"], atol=1e-13)


def test_golden_merge():
    for c in _golden("merge"):
        out, lse = oracle.merge_states(np.array(c["out_a"]), np.array(c["lse_a"]),
                                       np.array(c["out_b"]), np.array(c["lse_b"]))
        np.testing.assert_allclose(out, c["out"], atol=1e-13)
        assert abs(float(lse) - c["lse"]) < 1e-13


def test_golden_decode():
    for c in _golden("decode"):
        kp = _arr(c["k_pages"])
        vp = _arr(c["v_pages"])
        out, lse = oracle.decode_paged(np.array(c["q"]), kp, vp, np.array(c["block_table"]),
                                       np.array(c["kv_lens"]), c["scale"])
        np.testing.assert_allclose(out, c["out"], atol=1e-13)
        np.testing.assert_allclose(lse, c["lse"], atol=1e-13)


# ----------------------------------------------------------------------------- paging

def _case(seed, **kw):
    base = dict(batch=3, n_qo_heads=4, n_kv_heads=2, head_dim=8, page_size=4,
                kv_lens=[1, 9, 16], num_pages=20, dtype="f32")
    base.update(kw)
    return workloads.make_paged_decode(seed, **base)


def _np(case):
    return (case.q.double().numpy(), case.k_pages.double().numpy(), case.v_pages.double().numpy(),
            case.block_table.numpy(), case.kv_lens.numpy())


def check_gather_against_contiguous(gather):
    """Scatter a known contiguous K into pages and read it back through the table."""
    P, D, L = 4, 3, 10
    K = rng.normal(size=(L, D))
    V = rng.normal(size=(L, D))
    table = np.array([5, 1, 3], dtype=np.int32)
    kp = np.full((6, 1, P, D), np.nan)
    vp = np.full((6, 1, P, D), np.nan)
    for t in range(L):
        kp[table[t // P], 0, t % P] = K[t]
        vp[table[t // P], 0, t % P] = V[t]
    K2, V2 = gather(kp, vp, table, L, 0)
    return np.array_equal(K2, K) and np.array_equal(V2, V)


def test_gather_pins():
    assert check_gather_against_contiguous(oracle.gather_sequence)
    assert check_gather_against_contiguous(oracle.attention._gather_fast)


def check_page_shuffle_invariance(decode):
    c = _case(7)
    q, kp, vp, bt, lens = _np(c)
    out1, lse1 = decode(q, kp, vp, bt, lens, c.scale)
    perm = np.random.default_rng(3).permutation(kp.shape[0])      # new slot of each page
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    out2, lse2 = decode(q, kp2, vp2, bt2, lens, c.scale)
    return np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def check_poisoned_slots_unread(decode):
    c = _case(8)                     # unused pages and tail slots are NaN
    out, lse = decode(*_np(c), c.scale)
    return np.isfinite(out).all() and np.isfinite(lse).all()


def check_gqa_mapping(decode):
    """KV head g holds constant values g+1; query head h must read KV head h // G."""
    c = _case(9, n_qo_heads=6, n_kv_heads=3, kv_lens=[5, 2, 13])
    q, kp, vp, bt, lens = _np(c)
    for g in range(3):
        vp[:, g] = np.where(np.isnan(vp[:, g]), np.nan, g + 1.0)
    out, _ = decode(q, kp, vp, bt, lens, c.scale)
    want = np.repeat(np.arange(1.0, 4.0), 2)                       # heads 0,1 -> 1; 2,3 -> 2; 4,5 -> 3
    return np.allclose(out, want[None, :, None] * np.ones_like(out), atol=1e-13)


def check_decode_is_attention_over_logical_sequence(decode):
    """Rebuild each sequence from the pool with explicit loops and compare with attention on it."""
    c = _case(10)
    q, kp, vp, bt, lens = _np(c)
    out, lse = decode(q, kp, vp, bt, lens, c.scale)
    P = kp.shape[2]
    G = q.shape[1] // kp.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            L = int(lens[b])
            e = []
            for t in range(L):
                kt = kp[bt[b, t // P], h // G, t % P]
                e.append(math.exp(c.scale * math.fsum(q[b, h] * kt)))
            z = math.fsum(e)
            for d in range(q.shape[2]):
                ref = math.fsum(e[t] * vp[bt[b, t // P], h // G, t % P, d] for t in range(L)) / z
                if abs(out[b, h, d] - ref) > 1e-12:
                    return False
            if abs(lse[b, h] - math.log(z)) > 1e-12:
                return False
    return True


def check_empty_sequence(decode):
    c = _case(11, kv_lens=[0, 3, 0])
    out, lse = decode(*_np(c), c.scale)
    return (np.all(out[0] == 0) and np.all(lse[0] == -np.inf) and np.all(out[2] == 0)
            and np.isfinite(out[1]).all())


DECODE_PINS = [check_page_shuffle_invariance, check_poisoned_slots_unread, check_gqa_mapping,
               check_decode_is_attention_over_logical_sequence, check_empty_sequence]


@pytest.mark.parametrize("pin", DECODE_PINS, ids=lambda f: f.__name__)
def test_decode_pins(pin):
    assert pin(oracle.decode_paged)


def test_decode_rows_subset():
    c = _case(12)
    args = _np(c)
    full_o, full_l = oracle.decode_paged(*args, c.scale)
    rows = [(0, 1), (2, 3)]
    o, l = oracle.decode_paged(*args, c.scale, rows=rows)
    for b, h in rows:
        assert np.allclose(o[b, h], full_o[b, h], atol=1e-14) and abs(l[b, h] - full_l[b, h]) < 1e-14
    assert np.isnan(o[1, 0]).all()


# ----------------------------------------------------------------------------- prefill

def _prefill(seed, B=2, T=9, Hq=4, Hkv=2, D=8):
    c = workloads.make_prefill(seed, B, T, Hq, Hkv, D, dtype="f32")
    return c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), c.scale


def check_causal_row0(prefill):
    q, k, v, s = _prefill(1)
    out, lse = prefill(q, k, v, s)
    G = q.shape[2] // k.shape[2]
    for h in range(q.shape[2]):
        if not np.allclose(out[:, 0, h], v[:, 0, h // G], atol=1e-14):
            return False
        if not np.allclose(lse[:, h, 0], s * np.einsum("bd,bd->b", q[:, 0, h], k[:, 0, h // G]), atol=1e-13):
            return False
    return True


def check_causal_future_independence(prefill):
    """Row i must not change when keys/values after i change, and must change when key i does."""
    q, k, v, s = _prefill(2)
    out, _ = prefill(q, k, v, s)
    i = 4
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1:] += 5.0
    v2[:, i + 1:] -= 3.0
    out2, _ = prefill(q, k2, v2, s)
    k3 = k.copy()
    k3[:, i] += 2.0
    out3, _ = prefill(q, k3, v, s)
    return (np.array_equal(out[:, :i + 1], out2[:, :i + 1])
            and not np.allclose(out[:, i], out3[:, i]))


def check_last_row_is_full_attention(prefill):
    q, k, v, s = _prefill(3)
    out, lse = prefill(q, k, v, s)
    G = q.shape[2] // k.shape[2]
    T = q.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            e = [math.exp(s * math.fsum(q[b, T - 1, h] * k[b, j, h // G])) for j in range(T)]
            z = math.fsum(e)
            ref = [math.fsum(e[j] * v[b, j, h // G, d] for j in range(T)) / z for d in range(q.shape[3])]
            if not np.allclose(out[b, T - 1, h], ref, atol=1e-12) or abs(lse[b, h, T - 1] - math.log(z)) > 1e-12:
                return False
    return True


def check_prefill_middle_row_brute_force(prefill):
    q, k, v, s = _prefill(4)
    out, lse = prefill(q, k, v, s)
    b, h, i = 1, 3, 5
    G = q.shape[2] // k.shape[2]
    e = [math.exp(s * math.fsum(q[b, i, h] * k[b, j, h // G])) for j in range(i + 1)]
    z = math.fsum(e)
    ref = [math.fsum(e[j] * v[b, j, h // G, d] for j in range(i + 1)) / z for d in range(q.shape[3])]
    return np.allclose(out[b, i, h], ref, atol=1e-12) and abs(lse[b, h, i] - math.log(z)) < 1e-12


PREFILL_PINS = [check_causal_row0, check_causal_future_independence,
                check_last_row_is_full_attention, check_prefill_middle_row_brute_force]


@pytest.mark.parametrize("pin", PREFILL_PINS, ids=lambda f: f.__name__)
def test_prefill_pins(pin):
    assert pin(oracle.prefill_causal)


def test_prefill_rows_subset_matches_full():
    q, k, v, s = _prefill(5)
    full_o, full_l = oracle.prefill_causal(q, k, v, s)
    rows = [(0, 0, 0), (1, 2, 8), (0, 3, 4)]
    o, l = oracle.prefill_causal(q, k, v, s, rows=rows)
    for b, h, i in rows:
        np.testing.assert_allclose(o[b, i, h], full_o[b, i, h], atol=1e-13)
        assert abs(l[b, h, i] - full_l[b, h, i]) < 1e-13


# ----------------------------------------------------------------------------- merge / split

def check_split_merge_equals_unsplit(merge_many):
    c = _case(13, kv_lens=[1, 33, 64, 17], batch=4, num_pages=40)
    args = _np(c)
    ref_o, ref_l = oracle.decode_paged(*args, c.scale)
    for pps in (1, 2, 3, 7, 32):
        parts = oracle.decode_split_partials(*args, c.scale, pps)
        for b, (outs, lses) in enumerate(parts):
            o, l = merge_many(outs, lses)
            if not (np.allclose(o, ref_o[b], atol=1e-12) and np.allclose(l, ref_l[b], atol=1e-12)):
                return False
    return True


def check_merge_empty_side_is_identity(merge_many):
    o = rng.normal(size=(3, 5))
    l = rng.normal(size=3)
    mo, ml = merge_many(np.stack([o, np.zeros_like(o)]), np.stack([l, np.full(3, -np.inf)]))
    eo, el = merge_many(np.stack([np.zeros_like(o)] * 2), np.full((2, 3), -np.inf))
    return (np.allclose(mo, o, atol=1e-15) and np.allclose(ml, l, atol=1e-15)
            and np.all(eo == 0) and np.all(el == -np.inf))


def check_merge_two_single_keys(merge_many):
    """Two one-key states merge into the two-key closed form."""
    v1, v2 = rng.normal(size=4), rng.normal(size=4)
    s1, s2 = 0.8, -1.3
    mo, ml = merge_many(np.stack([v1[None], v2[None]]), np.array([[s1], [s2]]))
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    return np.allclose(mo[0], w1 * v1 + (1 - w1) * v2, atol=1e-14) and abs(ml[0] - math.log(math.exp(s1) + math.exp(s2))) < 1e-14


def check_merge_associative_commutative(merge_many):
    o = rng.normal(size=(3, 2, 4))
    l = rng.normal(size=(3, 2)) * 5
    ab_o, ab_l = merge_many(o[:2], l[:2])
    left = merge_many(np.stack([ab_o, o[2]]), np.stack([ab_l, l[2]]))
    bc_o, bc_l = merge_many(o[1:], l[1:])
    right = merge_many(np.stack([o[0], bc_o]), np.stack([l[0], bc_l]))
    rev = merge_many(o[::-1], l[::-1])
    return all(np.allclose(x[0], left[0], atol=1e-13) and np.allclose(x[1], left[1], atol=1e-13)
               for x in (right, rev))


MERGE_PINS = [check_split_merge_equals_unsplit, check_merge_empty_side_is_identity,
              check_merge_two_single_keys, check_merge_associative_commutative]


@pytest.mark.parametrize("pin", MERGE_PINS, ids=lambda f: f.__name__)
def test_merge_pins(pin):
    assert pin(oracle.merge_many)


def test_merge_states_pairwise_matches_many():
    o = rng.normal(size=(2, 3, 4))
    l = rng.normal(size=(2, 3))
    a = oracle.merge_states(o[0], l[0], o[1], l[1])
    b = oracle.merge_many(o, l)
    assert np.allclose(a[0], b[0]) and np.allclose(a[1], b[1])


def test_split_ranges():
    assert oracle.split_ranges(0, 4) == []
    assert oracle.split_ranges(5, 2) == [(0, 2), (2, 4), (4, 5)]
    assert oracle.split_ranges(4, 4) == [(0, 4)]


# ----------------------------------------------------------------------------- cascade

def _cascade(seed):
    return workloads.make_cascade(seed, n_requests=5, prefix_len=12, suffix_lens=[0, 1, 5, 9, 3],
                                  n_qo_heads=4, n_kv_heads=2, head_dim=8, page_size=4,
                                  num_pages=30, dtype="f32")


def test_cascade_equals_concatenated_decode():
    c = _cascade(21)
    args = (c.q.double().numpy(), c.k_pages.double().numpy(), c.v_pages.double().numpy())
    o, l = oracle.cascade_decode(*args, c.prefix_table.numpy(), c.prefix_len,
                                 c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)
    cc = c.concatenated()
    o2, l2 = oracle.decode_paged(*args, cc.block_table.numpy(), cc.kv_lens.numpy(), c.scale)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(l, l2, atol=1e-13)


def test_cascade_equals_merge_of_prefix_and_suffix():
    c = _cascade(22)
    q, kp, vp = c.q.double().numpy(), c.k_pages.double().numpy(), c.v_pages.double().numpy()
    o, l = oracle.cascade_decode(q, kp, vp, c.prefix_table.numpy(), c.prefix_len,
                                 c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)
    R = q.shape[0]
    pre_table = np.tile(c.prefix_table.numpy(), (R, 1))
    po, pl = oracle.decode_paged(q, kp, vp, pre_table, np.full(R, c.prefix_len), c.scale)
    so, sl = oracle.decode_paged(q, kp, vp, c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)
    mo, ml = oracle.merge_states(po, pl, so, sl)
    np.testing.assert_allclose(o, mo, atol=1e-13)
    np.testing.assert_allclose(l, ml, atol=1e-13)


# ----------------------------------------------------------------------------- unified max

def test_unified_max_equals_softmax():
    q = rng.normal(size=(3, 16))
    k = rng.normal(size=(50, 16)) * 2
    v = rng.normal(size=(50, 16))
    ref_o, ref_l = oracle.attend(q, k, v, 0.25)
    true_max = float((0.25 * q @ k.T).max())
    for phi in (true_max, true_max - 20.0, true_max + 20.0, 0.0):
        accs, ls = oracle.unified_max_partials(q, k, v, 0.25, phi, chunk=7)
        o, l = oracle.unified_max_combine(accs, ls, phi)
        np.testing.assert_allclose(o, ref_o, atol=1e-12)
        np.testing.assert_allclose(l, ref_l, atol=1e-12)


def test_unified_max_fallback_predicate():
    s = np.array([0.0, 1.0, 2.0])
    assert not oracle.unified_max_needs_fallback(s, 1.0, 60.0, 60.0)
    assert oracle.unified_max_needs_fallback(s, -70.0, 60.0, 60.0)      # 2 > -70 + 60
    assert oracle.unified_max_needs_fallback(s, 70.0, 60.0, 60.0)       # all < 70 - 60
    assert not oracle.unified_max_needs_fallback(np.array([]), 0.0, 60.0, 60.0)


# ----------------------------------------------------------------------------- planted mistakes

def _attend_mutant(kind):
    """Copies of the definition, each with one plausible slip."""
    def f(q, k, v, scale, keep=None):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        n = q.shape[0]
        if k.shape[0] == 0:
            return np.zeros((n, v.shape[1] if v.ndim == 2 else q.shape[1])), np.full(n, -np.inf)
        sc = 1.0 if kind == "no_scale" else scale
        s = sc * (q @ k.T)
        if keep is not None:
            s = np.where(keep, s, -np.inf)
        m = s.max(axis=1)
        if kind == "min_not_max":
            m = s.min(axis=1)
        e = np.exp(s - m[:, None]) if kind != "sign" else np.exp(m[:, None] - s)
        z = e.sum(axis=1)
        vv = k if kind == "k_for_v" else v
        out = e @ vv
        if kind != "no_normalise":
            out = out / z[:, None]
        lse = m + np.log(z)
        if kind == "lse_no_max":
            lse = np.log(z)
        return out, lse
    return f


@pytest.mark.parametrize("kind", ["no_scale", "sign", "k_for_v", "no_normalise", "lse_no_max",
                                  "min_not_max"])
def test_planted_mistakes_are_caught(kind):
    mutant = _attend_mutant(kind)
    failed = []
    for pin in ATTEND_PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin(mutant)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"mutant {kind} passed every pin"


def _decode_mutant(kind):
    def f(q, kp, vp, bt, lens, scale, rows=None):
        B, Hq, D = q.shape
        Hkv = kp.shape[1]
        G = Hq // Hkv
        P = kp.shape[2]
        out = np.zeros((B, Hq, D))
        lse = np.zeros((B, Hq))
        for b in range(B):
            for h in range(Hq):
                g = (h % Hkv) if kind == "gqa_modulo" else h // G
                L = int(lens[b]) + (1 if kind == "len_plus_one" else 0)
                idx = [(bt[b, t // P], t % P) if kind != "swap_page_slot" else (bt[b, t % P], t // P)
                       for t in range(L)]
                if kind == "identity_table":
                    idx = [(t // P, t % P) for t in range(L)]
                K = np.array([kp[p, g, sl] for p, sl in idx]).reshape(L, D)
                V = np.array([vp[p, g, sl] for p, sl in idx]).reshape(L, D)
                o, l = oracle.attend(q[b, h][None], K, V, scale)
                out[b, h], lse[b, h] = o[0], l[0]
        return out, lse
    return f


@pytest.mark.parametrize("kind", ["gqa_modulo", "len_plus_one", "swap_page_slot", "identity_table"])
def test_planted_decode_mistakes_are_caught(kind):
    mutant = _decode_mutant(kind)
    assert check_decode_is_attention_over_logical_sequence(_decode_mutant("none"))
    failed = []
    for pin in DECODE_PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin(mutant)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"decode mutant {kind} passed every pin"


def _prefill_mutant(kind):
    def f(q, k, v, scale, rows=None):
        B, T, Hq, D = q.shape
        G = Hq // k.shape[2]
        keep = np.tril(np.ones((T, T), dtype=bool), k=-1 if kind == "strict" else
                       (1 if kind == "plus_one" else 0))
        if kind == "no_mask":
            keep = np.ones((T, T), dtype=bool)
        out = np.zeros((B, T, Hq, D))
        lse = np.zeros((B, Hq, T))
        for b in range(B):
            for h in range(Hq):
                o, l = oracle.attend(q[b, :, h], k[b, :, h // G], v[b, :, h // G], scale, keep=keep)
                out[b, :, h], lse[b, h] = o, l
        return out, lse
    return f


@pytest.mark.parametrize("kind", ["strict", "plus_one", "no_mask"])
def test_planted_prefill_mistakes_are_caught(kind):
    mutant = _prefill_mutant(kind)
    failed = []
    for pin in PREFILL_PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin(mutant)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"prefill mutant {kind} passed every pin"


def _merge_mutant(kind):
    def f(outs, lses):
        outs, lses = np.asarray(outs, float), np.asarray(lses, float)
        M = lses.max(axis=0)
        fin = np.isfinite(M)
        Ms = np.where(fin, M, 0.0)
        w = np.where(np.isfinite(lses), np.exp(lses - Ms), 0.0)
        if kind == "unweighted":
            w = np.where(np.isfinite(lses), 1.0, 0.0)
        z = w.sum(axis=0)
        out = (w[..., None] * np.where(np.isfinite(lses)[..., None], outs, 0)).sum(axis=0)
        out = np.where(fin[..., None], out / np.where(fin, z, 1)[..., None], 0)
        lse = np.where(fin, (Ms + np.log(np.where(fin, z, 1))) if kind != "lse_max_only" else Ms, -np.inf)
        return out, lse
    return f


@pytest.mark.parametrize("kind", ["unweighted", "lse_max_only"])
def test_planted_merge_mistakes_are_caught(kind):
    mutant = _merge_mutant(kind)
    failed = [p.__name__ for p in MERGE_PINS if not p(mutant)]
    assert failed


# ----------------------------------------------------------------------------- workloads

def test_named_workload_shapes():
    c1 = workloads.single_seq_decode_f32()
    assert tuple(c1.q.shape) == (1, 8, 64) and c1.num_pages == 64 and c1.q.dtype.is_floating_point
    assert int(c1.kv_lens[0]) == 256 and c1.max_blocks == 16
    used = c1.block_table[0].tolist()
    assert len(set(used)) == 16 and all(0 <= p < 64 for p in used)


# ----------------------------------------------------------------------------- FP8 E4M3 pages

def check_e4m3_worked_values(f):
    # values fixed by the format: bias 7, 3 mantissa bits, subnormals at exponent 0,
    # NaN at exponent 15 / mantissa 7, no infinities
    want = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x30: 0.5, 0x7E: 448.0, 0x08: 2.0 ** -6,
            0x07: 7 * 2.0 ** -9, 0x01: 2.0 ** -9, 0xB8: -1.0, 0xFE: -448.0, 0x78: 256.0}
    v = f(np.array(list(want)))
    ok = np.array_equal(v, np.array(list(want.values())))
    neg_zero = f(np.array([0x80]))[0]
    return bool(ok and neg_zero == 0.0 and np.signbit(neg_zero) and np.isnan(f(np.array([0x7F, 0xFF]))).all())


def check_e4m3_matches_library(f):
    # every code against torch's float8_e4m3fn conversion (a library routine)
    torch = pytest.importorskip("torch")
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()
    v = f(np.arange(256))
    return bool(((v == lib) | (np.isnan(v) & np.isnan(lib))).all())


def check_e4m3_monotone_and_symmetric(f):
    pos = f(np.arange(0x7F))          # 0x00 .. 0x7E: every finite non-negative value
    neg = f(np.arange(0x80, 0xFF))
    return bool(np.all(np.diff(pos) > 0) and np.array_equal(neg, -pos))


FP8_VALUE_PINS = [check_e4m3_worked_values, check_e4m3_matches_library, check_e4m3_monotone_and_symmetric]


def _fp8_case(seed, B=3, Hq=8, Hkv=2, D=16, P=4, lens=(9, 1, 14), n_pages=12):
    r = np.random.default_rng(seed)
    codes_k = r.integers(0, 256, size=(n_pages, Hkv, P, D))
    codes_v = r.integers(0, 256, size=(n_pages, Hkv, P, D))
    # no NaN codes (exponent 15, mantissa 7) in real pages
    codes_k[(codes_k & 0x7F) == 0x7F] = 0x3F
    codes_v[(codes_v & 0x7F) == 0x7F] = 0x3F
    ks = r.uniform(1e-3, 2e-2, size=(n_pages, Hkv))
    vs = r.uniform(1e-3, 2e-2, size=(n_pages, Hkv))
    table = np.stack([r.permutation(n_pages)[:4] for _ in range(B)])
    q = r.normal(size=(B, Hq, D))
    return q, codes_k, codes_v, ks, vs, table, np.array(lens), 0.3


def check_fp8_decode_is_decode_of_dequantised_pages(f):
    # the dequantised pools are built here from torch's float8 conversion and the scales,
    # independently of the oracle's e4m3 function, then fed to the plain decode
    torch = pytest.importorskip("torch")
    q, ck, cv, ks, vs, table, lens, scale = _fp8_case(7)
    to_f = lambda c: torch.from_numpy(c.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    kf = to_f(ck) * ks[:, :, None, None]
    vf = to_f(cv) * vs[:, :, None, None]
    want = oracle.decode_paged(q, kf, vf, table, lens, scale)
    got = f(q, ck, cv, ks, vs, table, lens, scale)
    return np.allclose(got[0], want[0], atol=1e-12) and np.allclose(got[1], want[1], atol=1e-12)


def check_fp8_scale_invariances(f):
    # a common factor on every V scale scales the output; one on every K scale is the same
    # as a larger softmax scale
    q, ck, cv, ks, vs, table, lens, scale = _fp8_case(8)
    base = f(q, ck, cv, ks, vs, table, lens, scale)
    v3 = f(q, ck, cv, ks, vs * 3.0, table, lens, scale)
    k2 = f(q, ck, cv, ks * 2.0, vs, table, lens, scale)
    s2 = f(q, ck, cv, ks, vs, table, lens, scale * 2.0)
    return (np.allclose(v3[0], 3.0 * base[0], atol=1e-12) and np.allclose(v3[1], base[1], atol=1e-12)
            and np.allclose(k2[0], s2[0], atol=1e-12) and np.allclose(k2[1], s2[1], atol=1e-12))


def check_fp8_per_tile_scale(f):
    # doubling the scale of one (page, KV head) tile of V changes exactly the rows that read it
    q, ck, cv, ks, vs, table, lens, scale = _fp8_case(9)
    base = f(q, ck, cv, ks, vs, table, lens, scale)
    page = int(table[0, 0])
    vs2 = vs.copy()
    vs2[page, 1] *= 2.0
    got = f(q, ck, cv, ks, vs2, table, lens, scale)
    G = q.shape[1] // ck.shape[1]
    readers = {(b, h) for b in range(q.shape[0]) for h in range(q.shape[1])
               if h // G == 1 and page in set(table[b, : (lens[b] + 3) // 4].tolist())}
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            same = np.allclose(got[0][b, h], base[0][b, h], atol=1e-14)
            if same == ((b, h) in readers):
                return False
    return bool(readers)


FP8_DECODE_PINS = [check_fp8_decode_is_decode_of_dequantised_pages, check_fp8_scale_invariances,
                   check_fp8_per_tile_scale]


@pytest.mark.parametrize("pin", FP8_VALUE_PINS)
def test_e4m3_pins(pin):
    assert pin(oracle.e4m3_to_float)


@pytest.mark.parametrize("pin", FP8_DECODE_PINS)
def test_fp8_decode_pins(pin):
    assert pin(oracle.decode_paged_fp8)


def _e4m3_mutant(kind):
    def f(codes):
        c = np.asarray(codes).astype(np.int64) & 0xFF
        s, e, m = (c >> 7) & 1, (c >> 3) & 0xF, (c & 7).astype(np.float64)
        bias = 8 if kind == "bias" else 7
        if kind == "no_subnormal":
            mag = np.ldexp(1.0 + m / 8.0, e - bias)
        else:
            mag = np.where(e == 0, np.ldexp(m / 8.0, 1 - bias), np.ldexp(1.0 + m / 8.0, e - bias))
        if kind == "mantissa4":
            mag = np.where(e == 0, np.ldexp(m / 16.0, 1 - bias), np.ldexp(1.0 + m / 16.0, e - bias))
        val = mag if kind == "no_sign" else np.where(s == 1, -mag, mag)
        if kind != "no_nan":
            val = np.where((e == 15) & (c & 7 == 7), np.nan, val)
        return val
    return f


def _fp8_decode_mutant(kind):
    def f(q, ck, cv, ks, vs, table, lens, scale):
        if kind == "scale_transposed":
            ks2 = ks.copy()
            ks2[: ks.shape[1], :] = ks[: ks.shape[1], :][:, ::-1]
            ks = ks2
        if kind == "k_scale_for_v":
            vs = ks
        if kind == "page_not_logical":   # scale read by logical block index instead of page
            ks = np.roll(ks, 1, axis=0)
        return oracle.decode_paged_fp8(q, ck, cv, ks, vs, table, lens, scale)
    return f


@pytest.mark.parametrize("kind", ["bias", "no_subnormal", "mantissa4", "no_sign", "no_nan"])
def test_e4m3_planted_mistakes_are_caught(kind):
    assert not all(pin(_e4m3_mutant(kind)) for pin in FP8_VALUE_PINS)


@pytest.mark.parametrize("kind", ["scale_transposed", "k_scale_for_v", "page_not_logical"])
def test_fp8_decode_planted_mistakes_are_caught(kind):
    assert not all(pin(_fp8_decode_mutant(kind)) for pin in FP8_DECODE_PINS)


# ----------------------------------------------------------------------------- chunked paged prefill

def _chunk_case(seed, B=2, C=5, Hq=4, Hkv=2, D=8, P=4, prefix=(7, 0), n_pages=16):
    r = np.random.default_rng(seed)
    L = [L0 + C for L0 in prefix]
    nblk = [(l + P - 1) // P for l in L]
    order = r.permutation(n_pages)
    table = np.full((B, max(nblk)), -1)
    pos = 0
    for b in range(B):
        table[b, :nblk[b]] = order[pos:pos + nblk[b]]
        pos += nblk[b]
    # the sequences' K and V, contiguous, then scattered into the pool through the table
    ks = [r.normal(size=(l, Hkv, D)) for l in L]
    vs = [r.normal(size=(l, Hkv, D)) for l in L]
    kp = np.full((n_pages, Hkv, P, D), np.nan)
    vp = np.full((n_pages, Hkv, P, D), np.nan)
    for b in range(B):
        for t in range(L[b]):
            kp[table[b, t // P], :, t % P] = ks[b][t]
            vp[table[b, t // P], :, t % P] = vs[b][t]
    q = r.normal(size=(B, C, Hq, D))
    return q, kp, vp, table, np.array(prefix), ks, vs, 0.4


def check_chunk_without_prefix_is_causal_prefill(f):
    q, kp, vp, table, _, ks, vs, scale = _chunk_case(21, prefix=(0, 0))
    got = f(q, kp, vp, table, np.array([0, 0]), scale)
    want = oracle.prefill_causal(q, np.stack(ks), np.stack(vs), scale)
    return np.allclose(got[0], want[0], atol=1e-12) and np.allclose(got[1], want[1], atol=1e-12)


def check_single_token_chunk_is_decode(f):
    q, kp, vp, table, prefix, ks, vs, scale = _chunk_case(22, C=1, prefix=(9, 3))
    got = f(q, kp, vp, table, prefix, scale)
    want = oracle.decode_paged(q[:, 0], kp, vp, table, prefix + 1, scale)
    return np.allclose(got[0][:, 0], want[0], atol=1e-12) and np.allclose(got[1][:, :, 0], want[1], atol=1e-12)


def check_chunks_compose(f):
    # one chunk of 5 new tokens = a chunk of 2 followed by a chunk of 3
    q, kp, vp, table, prefix, ks, vs, scale = _chunk_case(23, C=5, prefix=(6, 1))
    whole = f(q, kp, vp, table, prefix, scale)
    first = f(q[:, :2], kp, vp, table, prefix, scale)
    second = f(q[:, 2:], kp, vp, table, prefix + 2, scale)
    return (np.allclose(whole[0][:, :2], first[0], atol=1e-12) and np.allclose(whole[0][:, 2:], second[0], atol=1e-12)
            and np.allclose(whole[1][:, :, :2], first[1], atol=1e-12) and np.allclose(whole[1][:, :, 2:], second[1], atol=1e-12))


def check_chunk_brute_force(f):
    q, kp, vp, table, prefix, ks, vs, scale = _chunk_case(24, B=1, C=3, Hq=2, Hkv=1, D=3, prefix=(4,))
    got = f(q, kp, vp, table, prefix, scale)
    L0 = int(prefix[0])
    for i in range(3):
        for h in range(2):
            sc = [scale * math.fsum(q[0, i, h, d] * ks[0][j][0][d] for d in range(3)) for j in range(L0 + i + 1)]
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            z = math.fsum(w)
            o = [math.fsum(w[j] * vs[0][j][0][d] for j in range(len(w))) / z for d in range(3)]
            if not (np.allclose(got[0][0, i, h], o, atol=1e-12) and abs(got[1][0, h, i] - (m + math.log(z))) < 1e-12):
                return False
    return True


def check_chunk_page_shuffle(f):
    q, kp, vp, table, prefix, ks, vs, scale = _chunk_case(25)
    perm = np.random.default_rng(5).permutation(kp.shape[0])
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    a = f(q, kp, vp, table, prefix, scale)
    b2 = f(q, kp2, vp2, table2, prefix, scale)
    return np.allclose(a[0], b2[0], atol=1e-13) and np.allclose(a[1], b2[1], atol=1e-13)


CHUNK_PINS = [check_chunk_without_prefix_is_causal_prefill, check_single_token_chunk_is_decode,
              check_chunks_compose, check_chunk_brute_force, check_chunk_page_shuffle]


@pytest.mark.parametrize("pin", CHUNK_PINS)
def test_prefill_paged_chunk_pins(pin):
    assert pin(oracle.prefill_paged_chunk)


def _chunk_mutant(kind):
    def f(q, kp, vp, table, prefix, scale):
        q = np.asarray(q, dtype=np.float64)
        B, C, Hq, D = q.shape
        Hkv = kp.shape[1]
        G = Hq // Hkv
        P = kp.shape[2]
        out = np.full((B, C, Hq, D), np.nan)
        lse = np.full((B, Hq, C), np.nan)
        for b in range(B):
            L0 = int(prefix[b])
            L = L0 + C
            lim = (L0 + np.arange(C)) if kind != "no_offset" else np.arange(C)
            keep = (np.arange(L)[None, :] < lim[:, None]) if kind == "strict" else (np.arange(L)[None, :] <= lim[:, None])
            tb = table[0] if kind == "first_table" else table[b]
            t = np.arange(L)
            pages = np.asarray(tb)[t // P]
            for h in range(Hq):
                g = h % Hkv if kind == "gqa_modulo" else h // G
                K = kp[pages, g, t % P]
                V = vp[pages, g, t % P]
                o, l = oracle.attend(q[b, :, h], K, V, scale, keep=keep)
                out[b, :, h] = o
                lse[b, h] = l
        return out, lse
    return f


@pytest.mark.parametrize("kind", ["strict", "no_offset", "first_table", "gqa_modulo"])
def test_prefill_paged_chunk_planted_mistakes_are_caught(kind):
    failed = []
    for pin in CHUNK_PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin(_chunk_mutant(kind))
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"mutant {kind} passed every pin"
