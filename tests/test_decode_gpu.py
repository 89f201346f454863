"""GPU parity of the paged decode path (attn_decode_paged, its unified-max variant and the
state merge) against the fp64 oracle, on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_28_gb300 import workloads
from tests._compare import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_28_gb300 import build
    build.build(quiet=True)
    from paged_kv_attention_28_gb300 import binding
    return binding


def to_dev(case):
    d = "cuda"
    return (case.q.to(d), case.k_pages.to(d), case.v_pages.to(d), case.block_table.to(d),
            case.kv_lens.to(d))


def run(b, case, num_splits=0, phi=None, dev=None, table=None, lens=None):
    q, kp, vp, bt, ln = dev if dev is not None else to_dev(case)
    if table is not None:
        bt = table.to("cuda")
    if lens is not None:
        ln = lens.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fb = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = b.decode_paged(q, kp, vp, bt, ln, case.scale, num_splits=num_splits, err_flag=err,
                              unified_phi=phi, fallback_count=fb)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item()), int(fb.item())


def ref(case, rows=None, table=None, lens=None):
    return oracle.decode_paged(case.q.double().numpy(), case.k_pages.float().numpy(),
                               case.v_pages.float().numpy(),
                               (case.block_table if table is None else table).numpy(),
                               (case.kv_lens if lens is None else lens).numpy(), case.scale, rows=rows)


def check(case, got, want, what):
    assert_close(got[0], want[0], case.dtype_name, what + " out")
    assert_close(got[1], want[1], case.dtype_name, what + " lse")


# ------------------------------------------------------------------------ named workloads

@pytest.mark.parametrize("splits", [1, 0, 4, 16])
def test_single_seq_decode_f32(b, splits):
    case = workloads.single_seq_decode_f32()
    got = run(b, case, splits)
    assert got[2] == 0
    check(case, got, ref(case), f"single_seq_decode_f32 splits={splits}")


def test_llama7b_batched_decode_all_rows(b):
    case = workloads.llama7b_batched_decode()
    dev = to_dev(case)
    want = ref(case)
    for splits in (0, 1, 8):
        got = run(b, case, splits, dev=dev)
        assert got[2] == 0
        check(case, got, want, f"llama7b_batched_decode splits={splits}")


def test_long_context_gqa_split32_all_rows(b):
    case = workloads.long_context_gqa_decode()
    dev = to_dev(case)
    want = ref(case)
    got = run(b, case, workloads.LONG_CONTEXT_SPLITS, dev=dev)
    assert got[2] == 0
    check(case, got, want, "long_context_gqa_decode splits=32")
    # the unified-max variant on the same data (wide logits): phi = 0 needs no fallback
    got_u = run(b, case, workloads.LONG_CONTEXT_SPLITS, phi=0.0, dev=dev)
    assert got_u[2] == 0 and got_u[3] == 0
    check(case, got_u, want, "long_context_gqa_decode unified phi=0")


# ------------------------------------------------------------------------ shape sweep

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_shapes(b, dtype, head_dim, group):
    hkv = 2
    lens = [1, 15, 16, 17, 100, 257, 0, 48]
    case = workloads.make_paged_decode(7 + group + head_dim, len(lens), hkv * group, hkv, head_dim,
                                       16, lens, num_pages=64, max_blocks=20, dtype=dtype,
                                       name=f"shapes {dtype} d{head_dim} g{group}")
    want = ref(case)
    dev = to_dev(case)
    for splits in (1, 3, 0):
        got = run(b, case, splits, dev=dev)
        assert got[2] == 0
        check(case, got, want, f"{case.name} splits={splits}")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 32])
def test_split_count_invariance(b, splits):
    case = workloads.make_paged_decode(31, 3, 8, 2, 128, 16, [1000, 513, 31], num_pages=160,
                                       max_blocks=64, dtype="bf16")
    got = run(b, case, splits)
    assert got[2] == 0
    check(case, got, ref(case), f"splits={splits}")


@pytest.mark.parametrize("dtype,head_dim,hq,hkv,splits", [
    ("f32", 64, 4, 4, 48), ("bf16", 128, 8, 8, 64), ("bf16", 128, 16, 4, 48)])
def test_many_splits_merge_in_rounds(b, dtype, head_dim, hq, hkv, splits):
    """More live splits than the merge's four warps take in one round (8 each): 43 to 64
    partials per row, so every warp loops and the last round is ragged; sequences of one
    split, of a few and of all are mixed."""
    case = workloads.make_paged_decode(40 + splits + head_dim, 4, hq, hkv, head_dim, 16,
                                       [4096, 700, 16, 3001], max_blocks=256, dtype=dtype)
    got = run(b, case, splits)
    assert got[2] == 0
    check(case, got, ref(case), f"{dtype} d{head_dim} {hq}/{hkv} splits={splits}")


def test_page_shuffle_invariance_gpu(b):
    case = workloads.make_paged_decode(32, 4, 8, 8, 64, 16, [70, 33, 160, 5], num_pages=40,
                                       dtype="f32")
    a1 = run(b, case, 2)
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(5))
    kp = torch.empty_like(case.k_pages)
    vp = torch.empty_like(case.v_pages)
    kp[perm] = case.k_pages
    vp[perm] = case.v_pages
    bt = torch.where(case.block_table >= 0, perm[case.block_table.clamp(min=0).long()].int(),
                     case.block_table)
    case2 = workloads.PagedDecodeCase(case.q, kp, vp, bt, case.kv_lens, case.scale)
    a2 = run(b, case2, 2)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1])


def test_empty_sequences(b):
    case = workloads.make_paged_decode(33, 3, 4, 4, 64, 16, [0, 5, 0], num_pages=8, max_blocks=4,
                                       dtype="f32")
    for splits in (1, 4):
        out, lse, err, _ = run(b, case, splits)
        assert err == 0
        assert np.all(out[0] == 0) and np.all(out[2] == 0)
        assert np.all(lse[0] == -np.inf) and np.all(lse[2] == -np.inf)
        check(case, (out, lse), ref(case), "empty")


# ------------------------------------------------------------------------ device-side checks

def test_bad_page_entry_sets_flag(b):
    case = workloads.make_paged_decode(34, 3, 4, 2, 64, 16, [40, 40, 40], num_pages=12,
                                       max_blocks=4, dtype="f32")
    table = case.block_table.clone()
    table[1, 1] = case.num_pages + 5               # out of range, inside the sequence
    table[2, 3] = 10**6                             # out of range but past the length: never read
    for splits in (1, 2):
        out, lse, err, _ = run(b, case, splits, table=table)
        assert err & b.PKV_DEVERR_BAD_PAGE
        assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
        want = ref(case, rows=[(bb, h) for bb in (0, 2) for h in range(4)])
        check(case, (out[[0, 2]], lse[[0, 2]]), (want[0][[0, 2]], want[1][[0, 2]]), "good rows")


def test_bad_length_sets_flag(b):
    case = workloads.make_paged_decode(35, 2, 4, 4, 64, 16, [20, 20], num_pages=8, max_blocks=2,
                                       dtype="f32")
    lens = case.kv_lens.clone()
    lens[0] = 2 * 16 + 1                            # above the table's capacity
    for splits in (1, 2):
        out, lse, err, _ = run(b, case, splits, lens=lens)
        assert err & b.PKV_DEVERR_BAD_LEN
        assert np.isnan(out[0]).all() and np.isnan(lse[0]).all()
        want = ref(case)
        check(case, (out[1:], lse[1:]), (want[0][1:], want[1][1:]), "good row")


# ------------------------------------------------------------------------ unified max

def _logits(case):
    q = case.q.double().numpy()
    out = []
    G = case.n_qo_heads // case.n_kv_heads
    for bb in range(case.batch):
        for h in range(case.n_qo_heads):
            K, _ = oracle.gather_sequence(case.k_pages.double().numpy(), case.v_pages.double().numpy(),
                                          case.block_table[bb].numpy(), int(case.kv_lens[bb]), h // G)
            out.append(case.scale * K @ q[bb, h])
    return out


@pytest.mark.parametrize("phi,expect_fallback", [(0.0, False), (-100.0, True), (200.0, True)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unified_max_matches_and_falls_back(b, phi, expect_fallback, dtype):
    case = workloads.make_paged_decode(36, 3, 8, 2, 128, 16, [300, 17, 64], num_pages=40,
                                       dtype=dtype, k_std=2.0)
    # the oracle's predicate says whether any row is unsafe against phi (beta = 60)
    unsafe = any(oracle.unified_max_needs_fallback(s, phi, 60.0, 60.0) for s in _logits(case))
    assert unsafe == expect_fallback
    want = ref(case)
    for splits in (1, 3):
        out, lse, err, fb = run(b, case, splits, phi=phi)
        assert err == 0
        assert (fb > 0) == expect_fallback
        check(case, (out, lse), want, f"unified phi={phi} splits={splits}")


def test_unified_max_single_hot_token_triggers_rescale(b):
    """One logit far above phi + 60 in the middle of a long sequence forces a raise."""
    case = workloads.make_paged_decode(37, 1, 4, 4, 64, 16, [400], num_pages=32, dtype="f32")
    kp = case.k_pages.clone()
    page = int(case.block_table[0, 12])
    kp[page, :, 5, :] = case.q[0, :, :] * 40.0      # q . k = 40 |q|^2 -> logit far above 60
    case2 = workloads.PagedDecodeCase(case.q, kp, case.v_pages, case.block_table, case.kv_lens,
                                      case.scale)
    out, lse, err, fb = run(b, case2, 1, phi=0.0)
    assert err == 0 and fb > 0
    check(case2, (out, lse), ref(case2), "hot token")


# ------------------------------------------------------------------------ merge

@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_states(b, out_dtype):
    g = torch.Generator().manual_seed(40)
    R, D = 37, 128
    oa, ob = torch.randn(R, D, generator=g), torch.randn(R, D, generator=g)
    la, lb = torch.randn(R, generator=g) * 5, torch.randn(R, generator=g) * 5
    la[3] = -math.inf
    lb[5] = -math.inf
    la[7] = lb[7] = -math.inf
    out, lse = b.merge_states(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    wo, wl = oracle.merge_states(oa.double().numpy(), la.double().numpy(), ob.double().numpy(),
                                 lb.double().numpy())
    name = "f32" if out_dtype == torch.float32 else "bf16"
    assert_close(out.float().cpu().numpy(), wo, name, "merge out")
    assert_close(lse.cpu().numpy(), wl, "f32", "merge lse")


def test_merge_states_in_place(b):
    g = torch.Generator().manual_seed(41)
    oa, ob = torch.randn(4, 8, 64, generator=g).cuda(), torch.randn(4, 8, 64, generator=g).cuda()
    la, lb = torch.randn(4, 8, generator=g).cuda(), torch.randn(4, 8, generator=g).cuda()
    wo, wl = oracle.merge_states(oa.double().cpu().numpy(), la.double().cpu().numpy(),
                                 ob.double().cpu().numpy(), lb.double().cpu().numpy())
    b.merge_states(oa, la, ob, lb, out=oa, lse=la)
    torch.cuda.synchronize()
    assert_close(oa.cpu().numpy(), wo, "f32", "in-place out")
    assert_close(la.cpu().numpy(), wl, "f32", "in-place lse")
