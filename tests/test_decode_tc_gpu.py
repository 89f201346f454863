"""GPU parity of the tensor-core GQA decode (bf16, head_dim 128, 4 or 8 query heads per KV
head) against the fp64 oracle, through attn_decode_paged.

Both products of the online softmax run on tcgen05 with the keys as the 128-row operand;
a tile is 8 pages of 16 keys. The cases cover tiles cut short by the sequence end or the
split end (whose slots past the end hold NaN in the pool), one-key and empty sequences,
split counts 1 to 32, the page-table and length checks, and a long-context batch of 8
query heads per KV head at full size. Tolerance: the bf16 bar of the other tests
("快速注意力内核与算子融合", Q&A on FlashAttention tiling; paged attention in the same
page's Q&A).
"""
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
    yield binding
    binding.debug_decode_stall(-1)


def run(b, case, splits, table=None, lens=None):
    d = "cuda"
    bt = (case.block_table if table is None else table).to(d)
    ln = (case.kv_lens if lens is None else lens).to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    out, lse = b.decode_paged(case.q.to(d), case.k_pages.to(d), case.v_pages.to(d), bt, ln, case.scale,
                              num_splits=splits, err_flag=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


def ref(case, rows=None, table=None, lens=None):
    return oracle.decode_paged(case.q.double().numpy(), case.k_pages.float().numpy(),
                               case.v_pages.float().numpy(),
                               (case.block_table if table is None else table).numpy(),
                               (case.kv_lens if lens is None else lens).numpy(), case.scale, rows=rows)


LENS = [1, 15, 16, 17, 127, 128, 129, 300, 1000, 2049, 0, 64]


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("splits", [1, 3, 0, 32])
def test_tc_decode_matches_oracle(b, G, splits):
    hkv = 2
    case = workloads.make_paged_decode(600 + G + splits, len(LENS), hkv * G, hkv, 128, 16, LENS, num_pages=400,
                                       max_blocks=140, dtype="bf16", k_std=1.5)
    out, lse, err = run(b, case, splits)
    assert err == 0
    want = ref(case)
    assert_close(out, want[0], "bf16", f"tc decode G={G} splits={splits} out")
    assert_close(lse, want[1], "bf16", f"tc decode G={G} splits={splits} lse")
    assert np.all(out[10] == 0) and np.all(lse[10] == -np.inf)   # the empty sequence


def test_tc_decode_one_split_longest_first_large_batch(b):
    """One split per sequence: the kernel hands out the sequences' units longest first (a
    counting sort in every CTA). 400 sequences (more than one per thread of the sort) of
    random lengths, including empty ones, one over the table's capacity and lengths past the
    last bucket; every row against the oracle."""
    rng = np.random.default_rng(681)
    lens = rng.integers(0, 700, size=400)
    lens[::37] = 0
    lens[5] = 8200                                   # 65 tiles: shares the first bucket
    case = workloads.make_paged_decode(681, 400, 8, 2, 128, 16, lens.tolist(),
                                       max_blocks=520, dtype="bf16")
    bad = case.kv_lens.clone()
    bad[7] = 520 * 16 + 1                            # above the table's capacity
    out, lse, err = run(b, case, 1, lens=bad)
    assert err & b.PKV_DEVERR_BAD_LEN
    assert np.isnan(out[7]).all() and np.isnan(lse[7]).all()
    keep = [i for i in range(400) if i != 7]
    want = ref(case, rows=[(bb, h) for bb in keep for h in range(8)], lens=bad)
    assert_close(out[keep], want[0][keep], "bf16", "longest-first out")
    assert_close(lse[keep], want[1][keep], "bf16", "longest-first lse")
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)   # an empty sequence


@pytest.mark.parametrize("splits", [4, 8])
def test_tc_decode_many_units_with_idle_splits(b, splits):
    """64 sequences x 8 KV heads x 4 or 8 splits: thousands of units, so running CTAs take
    many of them in turn, and short sequences leave most of their splits idle, so a CTA
    often passes several idle units between two live ones (the pipeline must neither stall
    nor wait out a bounded wait there). Every row against the oracle."""
    case = workloads.make_paged_decode(690 + splits, 64, 32, 8, 128, 16, (16, 1024), dtype="bf16")
    out, lse, err = run(b, case, splits)
    assert err == 0
    want = ref(case)
    assert_close(out, want[0], "bf16", f"idle splits S={splits} out")
    assert_close(lse, want[1], "bf16", f"idle splits S={splits} lse")


def test_tc_decode_wide_logits_move_the_max(b):
    """Keys scaled by 4 spread the logits so that later tiles raise the reference max."""
    case = workloads.make_paged_decode(640, 3, 32, 8, 128, 16, [3000, 900, 4096], num_pages=700,
                                       dtype="bf16", k_std=4.0)
    for splits in (1, 5):
        out, lse, err = run(b, case, splits)
        assert err == 0
        want = ref(case)
        assert_close(out, want[0], "bf16", f"wide logits splits={splits} out")
        assert_close(lse, want[1], "bf16", f"wide logits splits={splits} lse")


def test_tc_decode_bad_page_and_bad_length(b):
    case = workloads.make_paged_decode(650, 4, 16, 4, 128, 16, [200, 200, 200, 150], num_pages=60,
                                       max_blocks=16, dtype="bf16")
    table = case.block_table.clone()
    table[1, 3] = case.num_pages + 7                # inside sequence 1
    lens = case.kv_lens.clone()
    lens[2] = 16 * 16 + 1                           # above the table's capacity
    for splits in (1, 2):
        out, lse, err = run(b, case, splits, table=table, lens=lens)
        assert err & b.PKV_DEVERR_BAD_PAGE and err & b.PKV_DEVERR_BAD_LEN
        assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
        assert np.isnan(out[2]).all() and np.isnan(lse[2]).all()
        want = ref(case, rows=[(bb, h) for bb in (0, 3) for h in range(16)])
        assert_close(out[[0, 3]], want[0][[0, 3]], "bf16", "good rows out")
        assert_close(lse[[0, 3]], want[1][[0, 3]], "bf16", "good rows lse")


def test_long_context_gqa8_split32_sampled_rows(b):
    """The long-context batch with 8 query heads per KV head (64 over 8), 32 splits: every
    head of 6 KV groups against the oracle, and all rows finite."""
    case = workloads.long_context_gqa8_decode()
    out, lse, err = run(b, case, workloads.LONG_CONTEXT_SPLITS)
    assert err == 0
    rows = [(bb, h) for bb, g in [(0, 0), (1, 3), (2, 7), (3, 5), (0, 6), (3, 1)] for h in range(8 * g, 8 * g + 8)]
    want = ref(case, rows=rows)
    idx = tuple(np.array(rows).T)
    assert_close(out[idx], want[0][idx], "bf16", "gqa8 sampled out")
    assert_close(lse[idx], want[1][idx], "bf16", "gqa8 sampled lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_tc_decode_stalled_wait_is_reported_and_gpu_stays_usable(b):
    """The stall hook withholds one tile's K copies: the MMA warp's bounded wait runs out,
    the kernel reports it, writes the affected rows as NaN and returns; the next call matches."""
    case = workloads.make_paged_decode(660, 3, 8, 2, 128, 16, [300, 20, 520], num_pages=80, dtype="bf16")
    want = ref(case)
    b.debug_decode_stall(9, 200_000)  # the tile holding page 9 of each split
    try:
        out, lse, err = run(b, case, 1)
    finally:
        b.debug_decode_stall(-1)
    assert err & b.PKV_DEVERR_TIMEOUT
    assert np.isnan(out[[0, 2]]).all() and np.isnan(lse[[0, 2]]).all()   # 19 and 33 pages
    out, lse, err = run(b, case, 1)
    assert err == 0
    assert_close(out, want[0], "bf16", "after a timed-out launch out")
    assert_close(lse, want[1], "bf16", "after a timed-out launch lse")


@pytest.mark.parametrize("G", [4, 8])
def test_tc_unified_max_hot_token_and_presets(b, G):
    """FlashDecoding++'s unified maximum on the tensor-core path: with phi = 0 a planted key
    whose logit lies far above phi + 60 forces a raise (counted); presets far above or below
    every logit fall back on the first tile; every result matches the oracle."""
    case = workloads.make_paged_decode(670 + G, 2, 2 * G, 2, 128, 16, [700, 333], num_pages=80, dtype="bf16")
    kp = case.k_pages.clone()
    page = int(case.block_table[0, 20])
    kp[page, 0, 3, :] = (case.q[0, 0, :].float() * 30.0).to(torch.bfloat16)  # q.k/sqrt(d) ~ 30 |q|^2/11
    c2 = workloads.PagedDecodeCase(case.q, kp, case.v_pages, case.block_table, case.kv_lens, case.scale)
    want = ref(c2)
    d = "cuda"
    for phi, expect in ((0.0, True), (0.0, True), (-200.0, True), (300.0, True)):
        err = torch.zeros(1, dtype=torch.int32, device=d)
        fb = torch.zeros(1, dtype=torch.int32, device=d)
        out, lse = b.decode_paged(c2.q.to(d), c2.k_pages.to(d), c2.v_pages.to(d), c2.block_table.to(d),
                                  c2.kv_lens.to(d), c2.scale, num_splits=2, err_flag=err, unified_phi=phi,
                                  fallback_count=fb)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert (int(fb.item()) > 0) == expect
        assert_close(out.float().cpu().numpy(), want[0], "bf16", f"unified phi={phi} out")
        assert_close(lse.cpu().numpy(), want[1], "bf16", f"unified phi={phi} lse")
    # without the planted key and with phi near the logits, no fallback happens
    err = torch.zeros(1, dtype=torch.int32, device=d)
    fb = torch.zeros(1, dtype=torch.int32, device=d)
    out, lse = b.decode_paged(case.q.to(d), case.k_pages.to(d), case.v_pages.to(d), case.block_table.to(d),
                              case.kv_lens.to(d), case.scale, num_splits=2, err_flag=err, unified_phi=0.0,
                              fallback_count=fb)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(fb.item()) == 0
    want = ref(case)
    assert_close(out.float().cpu().numpy(), want[0], "bf16", "unified no fallback out")
    assert_close(lse.cpu().numpy(), want[1], "bf16", "unified no fallback lse")
