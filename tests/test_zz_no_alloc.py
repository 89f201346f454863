"""The allocation-free decode entry point, attn_decode_paged_noalloc, checked against
attn_decode_paged through the C ABI.

Some callers cannot allocate device memory when they call in: an inference
runtime's enqueue hook that may not allocate while it runs, or a process that
reserved all device memory for its own pool up front. For them the library
keeps split partial states in its own static device scratch array. This file's
name makes pytest collect it last.
"""
import ctypes

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


def _noalloc(b, case, dev, splits):
    q, kp, vp, bt, ln = dev
    out = torch.full_like(q, float("nan"))
    lse = torch.full((case.batch, case.n_qo_heads), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = b.lib.attn_decode_paged_noalloc(
        p(q), p(kp), p(vp), p(bt), p(ln), p(out), p(lse), case.batch, case.max_blocks,
        case.num_pages, case.n_qo_heads, case.n_kv_heads, case.head_dim, case.page_size,
        case.scale, splits, b.PKV_BF16 if case.dtype_name == "bf16" else b.PKV_F32, p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, out, lse, int(err.item())


def test_noalloc_matches_workspace_entry_point_on_two_calls(b):
    cases = [
        (workloads.make_paged_decode(71, 4, 16, 4, 128, 16, [1500, 700, 2048, 33], num_pages=400,
                                     max_blocks=128, dtype="bf16"), 8),
        (workloads.make_paged_decode(72, 3, 8, 8, 64, 16, [300, 17, 64], num_pages=40,
                                     max_blocks=32, dtype="f32"), 4),
    ]
    for case, splits in cases:                     # two calls in a row, different shapes
        dev = tuple(t.to("cuda") for t in (case.q, case.k_pages, case.v_pages, case.block_table,
                                           case.kv_lens))
        assert b.decode_workspace_size(case.batch, case.max_blocks, case.n_qo_heads,
                                       case.n_kv_heads, case.head_dim, case.page_size, splits,
                                       b._dt(case.q)) > 0   # the scratch array is really used
        want_o, want_l = b.decode_paged(*dev, case.scale, num_splits=splits)
        torch.cuda.synchronize()
        rc, out, lse, err = _noalloc(b, case, dev, splits)
        assert rc == b.PKV_OK and err == 0
        assert_close(out.float().cpu().numpy(), want_o.float().cpu().numpy(), case.dtype_name,
                     "noalloc out")
        assert_close(lse.cpu().numpy(), want_l.cpu().numpy(), case.dtype_name, "noalloc lse")


def test_noalloc_rejects_shapes_beyond_the_scratch_limit(b):
    # 64 sequences x 64 heads x 64 splits of 128-wide fp32 partials is ~134 MB > 8 MiB
    case = workloads.make_paged_decode(73, 64, 64, 64, 128, 16, [0] * 64, num_pages=64,
                                       max_blocks=64, dtype="bf16")
    need = b.decode_workspace_size(64, 64, 64, 64, 128, 16, 64, b.PKV_BF16)
    assert need > (8 << 20)
    dev = tuple(t.to("cuda") for t in (case.q, case.k_pages, case.v_pages, case.block_table,
                                       case.kv_lens))
    rc, _, _, _ = _noalloc(b, case, dev, 64)
    assert rc == b.PKV_ERR_WORKSPACE


def test_noalloc_call_allocates_no_device_memory_and_matches_the_oracle(b):
    """With its inputs and outputs already in place, a call leaves the device's free memory
    unchanged (it allocates nothing, and the scratch array was in place since load time),
    and its result is the fp64 oracle's."""
    case = workloads.make_paged_decode(74, 4, 16, 4, 128, 16, [1500, 700, 2048, 33], num_pages=400,
                                       max_blocks=128, dtype="bf16")
    q, kp, vp, bt, ln = (t.to("cuda") for t in (case.q, case.k_pages, case.v_pages, case.block_table,
                                               case.kv_lens))
    out = torch.empty_like(q)
    lse = torch.empty((case.batch, case.n_qo_heads), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        return b.lib.attn_decode_paged_noalloc(
            p(q), p(kp), p(vp), p(bt), p(ln), p(out), p(lse), case.batch, case.max_blocks,
            case.num_pages, case.n_qo_heads, case.n_kv_heads, case.head_dim, case.page_size,
            case.scale, 8, b.PKV_BF16, p(err), stream)

    assert call() == b.PKV_OK                       # first call on the device: address lookup
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert call() == b.PKV_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert int(err.item()) == 0
    want_o, want_l = oracle.decode_paged(case.q.double().numpy(), case.k_pages.float().numpy(),
                                         case.v_pages.float().numpy(), case.block_table.numpy(),
                                         case.kv_lens.numpy(), case.scale)
    assert_close(out.float().cpu().numpy(), want_o, "bf16", "noalloc out vs oracle")
    assert_close(lse.cpu().numpy(), want_l, "bf16", "noalloc lse vs oracle")
