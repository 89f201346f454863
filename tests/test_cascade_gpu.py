"""GPU parity of attn_decode_cascade (shared prefix once + suffix + merge) against the
oracle's definition: plain attention over each request's prefix + suffix."""
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


def run(b, c, prefix_table=None):
    d = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pt = c.prefix_table if prefix_table is None else prefix_table
    out, lse = b.decode_cascade(c.q.to(d), c.k_pages.to(d), c.v_pages.to(d), pt.to(d), c.prefix_len,
                                c.suffix_table.to(d), c.suffix_lens.to(d), c.scale, err_flag=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


def ref(c):
    return oracle.cascade_decode(c.q.double().numpy(), c.k_pages.float().numpy(),
                                 c.v_pages.float().numpy(), c.prefix_table.numpy(), c.prefix_len,
                                 c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)


@pytest.mark.parametrize("R,prefix,suffix,Hq,Hkv", [
    (6, 64, [0, 5, 40, 17, 64, 3], 8, 2),       # prefix of 4 pages: one partial key tile
    (5, 48, [1, 16, 17, 100, 0], 8, 8),         # G = 1
    (9, 256, [33, 2, 0, 77, 128, 5, 9, 300, 16], 16, 2),  # G = 8, two full key tiles
    (100, 160, (1, 200), 32, 8),                # 400 query rows: two row pairs, ragged
    (4, 0, [10, 20, 30, 40], 8, 2),             # no prefix at all
])
def test_cascade_small(b, R, prefix, suffix, Hq, Hkv):
    c = workloads.make_cascade(80 + R + prefix, R, prefix, suffix, Hq, Hkv, 128, page_size=16,
                               num_pages=None, dtype="bf16")
    out, lse, err = run(b, c)
    assert err == 0
    wo, wl = ref(c)
    assert_close(out, wo, "bf16", f"cascade R={R} prefix={prefix} out")
    assert_close(lse, wl, "bf16", f"cascade R={R} prefix={prefix} lse")


def test_cascade_shared_prefix_decode_all_rows(b):
    c = workloads.cascade_shared_prefix_decode()
    out, lse, err = run(b, c)
    assert err == 0
    wo, wl = ref(c)
    assert_close(out, wo, "bf16", "cascade_shared_prefix_decode out")
    assert_close(lse, wl, "bf16", "cascade_shared_prefix_decode lse")
    # the same cache as concatenated sequences through the plain decode path agrees too
    cc = c.concatenated()
    d = "cuda"
    o2, l2 = b.decode_paged(cc.q.to(d), cc.k_pages.to(d), cc.v_pages.to(d), cc.block_table.to(d),
                            cc.kv_lens.to(d), cc.scale)
    torch.cuda.synchronize()
    assert_close(out, o2.float().cpu().numpy(), "bf16", "cascade vs concatenated decode")


def test_cascade_bad_prefix_page_sets_flag(b):
    c = workloads.make_cascade(90, 4, 64, [8, 8, 8, 8], 8, 2, 128, page_size=16, dtype="bf16")
    pt = c.prefix_table.clone()
    pt[2] = c.num_pages + 3
    out, lse, err = run(b, c, prefix_table=pt)
    assert err & b.PKV_DEVERR_BAD_PAGE
    assert np.isnan(out).all() and np.isnan(lse).all()
