"""GPU parity of attn_decode_paged_fp8 (E4M3 page pools with per-(page, KV head) scales)
against the fp64 oracle's decode over the dequantised pages, on the same seeded codes."""
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


def to_dev(c):
    return tuple(t.to("cuda") for t in (c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                        c.block_table, c.kv_lens))


def run(b, c, splits=0, dev=None, table=None):
    q, kc, vc, ks, vs, bt, ln = dev if dev is not None else to_dev(c)
    if table is not None:
        bt = table.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = b.decode_paged_fp8(q, kc, vc, ks, vs, bt, ln, c.scale, num_splits=splits, err_flag=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


def ref(c, rows=None, table=None):
    return oracle.decode_paged_fp8(c.q.double().numpy(), c.k_codes.numpy(), c.v_codes.numpy(),
                                   c.k_scale.numpy(), c.v_scale.numpy(),
                                   (c.block_table if table is None else table).numpy(),
                                   c.kv_lens.numpy(), c.scale, rows=rows)


def check(got, want, what):
    assert_close(got[0], want[0], "bf16", what + " out")
    assert_close(got[1], want[1], "bf16", what + " lse")


def test_llama7b_batched_decode_fp8_all_rows(b):
    c = workloads.llama7b_batched_decode_fp8()
    dev = to_dev(c)
    want = ref(c)
    for splits in (0, 1, 8):
        got = run(b, c, splits, dev=dev)
        assert got[2] == 0
        check(got, want, f"llama7b_batched_decode_fp8 splits={splits}")


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_fp8_shapes(b, head_dim, group):
    hkv = 2
    lens = [1, 15, 16, 17, 100, 257, 0, 48]
    c = workloads.make_paged_decode_fp8(70 + group + head_dim, len(lens), hkv * group, hkv, head_dim,
                                        16, lens, num_pages=64, max_blocks=20)
    want = ref(c)
    for splits in (0, 1, 3):
        got = run(b, c, splits)
        assert got[2] == 0
        check(got, want, f"fp8 D={head_dim} G={group} splits={splits}")


def test_decode_fp8_wide_scales_and_logits(b):
    # k ~ 3 N(0,1) spreads the logits; the per-tile scales then span a wide range too
    c = workloads.make_paged_decode_fp8(71, 4, 32, 8, 128, 16, [3000, 1, 700, 2049], num_pages=512,
                                        k_std=3.0, v_std=0.5)
    want = ref(c)
    for splits in (0, 16):
        got = run(b, c, splits)
        assert got[2] == 0
        check(got, want, f"fp8 wide splits={splits}")


@pytest.mark.parametrize("head_dim", [64, 128])
def test_decode_fp8_bad_page_sets_flag(b, head_dim):
    c = workloads.make_paged_decode_fp8(72, 3, 4, 2, head_dim, 16, [40, 40, 40], num_pages=12, max_blocks=4)
    table = c.block_table.clone()
    table[1, 1] = c.num_pages + 5               # out of range, inside the sequence
    table[2, 3] = 10**6                         # out of range but past the length: never read
    for splits in (1, 2):
        out, lse, err = run(b, c, splits, table=table)
        assert err & b.PKV_DEVERR_BAD_PAGE
        assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
        want = ref(c, rows=[(bb, h) for bb in (0, 2) for h in range(4)], table=table)
        check((out[[0, 2]], lse[[0, 2]]), (want[0][[0, 2]], want[1][[0, 2]]), "fp8 good rows")


def test_decode_fp8_tensor_core_many_units_and_idle_splits(b):
    """head_dim 128 runs on the tensor cores: 48 sequences x 4 KV heads x 6 splits, so CTAs
    take many units in turn, with short sequences leaving most splits idle; and one split
    per sequence (the longest-first order). Every row against the oracle."""
    c = workloads.make_paged_decode_fp8(74, 48, 16, 4, 128, 16, (1, 1500), k_std=2.0)
    want = ref(c)
    for splits in (6, 1):
        got = run(b, c, splits)
        assert got[2] == 0
        check(got, want, f"fp8 tensor cores splits={splits}")


def test_decode_fp8_rejects_missing_scales(b):
    c = workloads.make_paged_decode_fp8(73, 1, 4, 4, 64, 16, [20], num_pages=4)
    q, kc, vc, ks, vs, bt, ln = to_dev(c)
    L = b.lib
    p = lambda t: None if t is None else __import__("ctypes").c_void_p(t.data_ptr())
    st = L.attn_decode_paged_fp8(p(q), p(kc), p(vc), None, p(vs), p(bt), p(ln), p(q), None, 1,
                                 bt.shape[1], c.num_pages, 4, 4, 64, 16, c.scale, 1, None, 0, None,
                                 None)
    assert st == b.PKV_ERR_INVALID_ARG


@pytest.mark.parametrize("q_mag", [3e5, 1e-7])
@pytest.mark.parametrize("G", [1, 4])
def test_fp8_query_far_outside_f16_range(b, q_mag, G):
    """The kernel takes q through f16 after scaling each head by a power of two: queries
    whose magnitudes lie far above f16's largest value (65504) or below its smallest
    normal give the same attention as the oracle's. The softmax scale shrinks or grows by
    the same factor, so the logits keep the workload's spread."""
    c = workloads.make_paged_decode_fp8(120 + G, 3, 4 * G, 4, 128, 16, [300, 77, 512], q_std=q_mag,
                                        scale=1.0 / (q_mag * 128 ** 0.5))
    assert float(c.q.float().abs().max()) > 65504 or float(c.q.float().abs().max()) < 6.1e-5
    got = run(b, c, 2)
    assert got[2] == 0
    check(got, ref(c), f"fp8 q magnitude {q_mag} G={G}")


def test_long_context_gqa8_fp8_split32_sampled_rows(b):
    """The long-context batch with 8 query heads per KV head over E4M3 pools (the tensor-core
    path, codes converted to f16 in shared memory), 32 splits: every head of 6 KV groups
    against the oracle, and all rows finite."""
    c = workloads.long_context_gqa8_decode_fp8()
    got = run(b, c, 32)
    assert got[2] == 0
    rows = [(bb, h) for bb, g in [(0, 0), (1, 3), (2, 7), (3, 5), (0, 6), (3, 1)] for h in range(8 * g, 8 * g + 8)]
    want = ref(c, rows=rows)
    idx = tuple(np.array(rows).T)
    check((got[0][idx], got[1][idx]), (want[0][idx], want[1][idx]), "fp8 gqa8 sampled")
    assert np.isfinite(got[0]).all() and np.isfinite(got[1]).all()


def test_fp8_tensor_core_stalled_wait_is_reported_and_gpu_stays_usable(b):
    """The stall hook withholds the K copies of the tile holding page 9 of each split on the
    E4M3 tensor-core path (4 query heads per KV head): the converters' bounded wait runs out,
    the kernel reports it and writes the affected rows as NaN; the next call matches."""
    c = workloads.make_paged_decode_fp8(661, 3, 8, 2, 128, 16, [300, 20, 520], num_pages=80)
    want = ref(c)
    b.debug_decode_stall(9, 200_000)
    try:
        out, lse, err = run(b, c, 1)
    finally:
        b.debug_decode_stall(-1)
    assert err & b.PKV_DEVERR_TIMEOUT
    assert np.isnan(out[[0, 2]]).all() and np.isnan(lse[[0, 2]]).all()   # 19 and 33 pages
    got = run(b, c, 1)
    assert got[2] == 0
    check(got, want, "fp8 after a timed-out launch")

