"""Failure handling on the GPU, without a fault: a bounded wait inside the decode kernel
is made to run out, and the test checks that the kernel reports it and that the GPU
stays usable.

``attn_debug_decode_stall(page, limit)`` makes the producer warp of every decode CTA
withhold one page's copies (and the arrival that announces them), with a short limit on
every pipeline wait. The consumer waiting for that page gives up: the kernel ORs
PKV_DEVERR_TIMEOUT into the error flag, waits (bounded) for the copies it did issue,
writes that CTA's rows as NaN and returns. CTAs whose split has no such page are not
affected. A normal call afterwards, on the same stream, must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_28_gb300 import workloads
from tests._compare import assert_close

pytestmark = pytest.mark.gpu

LIMIT_NS = 200_000  # 0.2 ms per wait


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_28_gb300 import build
    build.build(quiet=True)
    from paged_kv_attention_28_gb300 import binding
    yield binding
    binding.debug_decode_stall(-1)


def _call(b, c, d, splits, unified=False):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(unified_phi=0.0) if unified else {}
    out, lse = b.decode_paged(*d, c.scale, num_splits=splits, err_flag=err, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("splits,unified", [(1, False), (3, False), (1, True)])
def test_decode_wait_that_runs_out_is_reported_and_gpu_stays_usable(b, splits, unified):
    # lengths 300, 20 and 520 tokens: 19, 2 and 33 pages
    c = workloads.make_paged_decode(77, 3, 8, 8, 128, 16, [300, 20, 520], num_pages=80, dtype="bf16")
    d = tuple(t.cuda() for t in (c.q, c.k_pages, c.v_pages, c.block_table, c.kv_lens))
    want_o, want_l = oracle.decode_paged(c.q.double().numpy(), c.k_pages.float().numpy(),
                                         c.v_pages.float().numpy(), c.block_table.numpy(),
                                         c.kv_lens.numpy(), c.scale)
    b.debug_decode_stall(2, LIMIT_NS)  # the third page of every split
    try:
        out, lse, err = _call(b, c, d, splits, unified)
    finally:
        b.debug_decode_stall(-1)
    assert err & b.PKV_DEVERR_TIMEOUT
    # sequences 0 and 2 have a third page in (at least) their first split: their rows are NaN
    assert np.isnan(out[[0, 2]]).all() and np.isnan(lse[[0, 2]]).all()
    # sequence 1 has two pages: no CTA of it waits for a withheld page
    assert_close(out[1], want_o[1], "bf16", "unaffected sequence out")
    assert_close(lse[1], want_l[1], "bf16", "unaffected sequence lse")
    # the context is intact: the same call again, with no stall, matches the oracle
    out, lse, err = _call(b, c, d, splits, unified)
    assert err == 0
    assert_close(out, want_o, "bf16", "decode after a timed-out launch, out")
    assert_close(lse, want_l, "bf16", "decode after a timed-out launch, lse")


def test_stall_hook_rejects_bad_arguments(b):
    assert b.lib.attn_debug_decode_stall(-2, 0) == b.PKV_ERR_INVALID_ARG
    assert b.lib.attn_debug_decode_stall(0, 20_000_000_000) == b.PKV_ERR_INVALID_ARG
    assert b.lib.attn_debug_decode_stall(-1, 0) == b.PKV_OK
