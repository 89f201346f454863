"""The C-ABI library loads on a machine without a GPU and exports what the header declares.

No compute call is made here. Only host-side argument checking, split planning
and workspace sizing run, and every call shown returns before any launch.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv_attn.h")


@pytest.fixture(scope="module")
def b():
    from paged_kv_attention_28_gb300 import build
    build.build(quiet=True)
    from paged_kv_attention_28_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(b):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(b.lib, n), n
    assert sorted(b.EXPORTS) == names


def test_status_strings(b):
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(b.status_string(code), str) and b.status_string(code)


def test_split_planning(b):
    # explicit request: 2048 pages in 32 splits of 64 pages
    assert b.decode_num_splits(4, 2048, 32, 8, 128, 16, 32) == 32
    # a request above the page count is capped
    assert b.decode_num_splits(1, 4, 8, 8, 64, 16, 100) == 4
    # uneven: 10 pages in 3 splits -> 4 pages per split -> 3 splits
    assert b.decode_num_splits(1, 10, 8, 8, 64, 16, 3) == 3
    # 10 pages in 4 splits -> 3 pages per split -> 4 splits
    assert b.decode_num_splits(1, 10, 8, 8, 64, 16, 4) == 4
    # automatic choice: between 1 and 64 splits, at most one per page
    for args in [(16, 256, 32, 32, 128, 16), (1, 16, 8, 8, 64, 16), (4, 2048, 32, 8, 128, 16),
                 (64, 8, 8, 8, 64, 16)]:
        s = b.decode_num_splits(*args, 0)
        assert 1 <= s <= min(64, args[1])
    # a large batch of long sequences already fills the GPU: few splits
    assert b.decode_num_splits(512, 256, 32, 32, 128, 16, 0) <= 2


def test_workspace_size(b):
    assert b.decode_workspace_size(1, 16, 8, 8, 64, 16, 1) == 0
    # the query and the planner agree for both dtypes
    # layout: partial O [rows][S][D] fp32, then partial LSE [rows][S] fp32 on a 256-byte boundary
    up = lambda x: (x + 255) // 256 * 256
    for dt in (b.PKV_F32, b.PKV_BF16):
        s = b.decode_num_splits(16, 256, 32, 32, 128, 16, 0, dt)
        n = b.decode_workspace_size(16, 256, 32, 32, 128, 16, 0, dt)
        rows = 16 * 32
        assert n == (0 if s == 1 else rows * s * 128 * 4 + up(rows * s * 4))
    n = b.decode_workspace_size(4, 2048, 32, 8, 128, 16, 32)
    rows = 4 * 32
    assert n == rows * 32 * 128 * 4 + up(rows * 32 * 4)
    with pytest.raises(b.AttnError):
        b.decode_workspace_size(1, 0, 8, 8, 64, 16, 1)
    with pytest.raises(b.AttnError):
        b.decode_workspace_size(1, 16, 6, 4, 64, 16, 1)


def test_invalid_arguments_rejected_before_launch(b):
    L = b.lib
    nul = None
    # null pointers with a non-empty batch
    assert L.attn_decode_paged(nul, nul, nul, nul, nul, nul, nul, 1, 1, 1, 8, 8, 64, 16, 1.0, 0,
                               b.PKV_F32, nul, 0, nul, nul) == b.PKV_ERR_INVALID_ARG
    # heads not a multiple
    assert L.attn_decode_paged(nul, nul, nul, nul, nul, nul, nul, 1, 1, 1, 6, 4, 64, 16, 1.0, 0,
                               b.PKV_F32, nul, 0, nul, nul) == b.PKV_ERR_INVALID_ARG
    # bad dtype
    assert L.attn_decode_paged(nul, nul, nul, nul, nul, nul, nul, 1, 1, 1, 8, 8, 64, 16, 1.0, 0,
                               9, nul, 0, nul, nul) == b.PKV_ERR_INVALID_ARG
    # non-finite scale
    assert L.attn_decode_paged(nul, nul, nul, nul, nul, nul, nul, 1, 1, 1, 8, 8, 64, 16,
                               float("nan"), 0, b.PKV_F32, nul, 0, nul, nul) == b.PKV_ERR_INVALID_ARG
    # an empty batch is a no-op
    assert L.attn_decode_paged(nul, nul, nul, nul, nul, nul, nul, 0, 1, 1, 8, 8, 64, 16, 1.0, 0,
                               b.PKV_F32, nul, 0, nul, nul) == b.PKV_OK
    assert L.attn_merge_states(nul, nul, nul, nul, nul, nul, 0, 64, b.PKV_F32, nul) == b.PKV_OK
    assert L.attn_merge_states(nul, nul, nul, nul, nul, nul, 3, 64, b.PKV_F32, nul) == b.PKV_ERR_INVALID_ARG
    assert L.attn_prefill_causal(nul, nul, nul, nul, nul, 0, 16, 8, 8, 128, 1.0, b.PKV_BF16, nul,
                                 nul) == b.PKV_OK
    assert L.attn_prefill_causal(nul, nul, nul, nul, nul, 1, 16, 8, 8, 128, 1.0, b.PKV_BF16, nul,
                                 nul) == b.PKV_ERR_INVALID_ARG


def test_unsupported_shapes_are_reported(b):
    # pointers that are aligned but never dereferenced: UNSUPPORTED is returned first
    p = ctypes.c_void_p(1 << 20)
    L = b.lib
    assert L.attn_decode_paged(p, p, p, p, p, p, p, 1, 1, 1, 8, 8, 96, 16, 1.0, 1, b.PKV_F32,
                               None, 0, None, None) == b.PKV_ERR_UNSUPPORTED
    assert L.attn_decode_paged(p, p, p, p, p, p, p, 1, 1, 1, 8, 8, 64, 32, 1.0, 1, b.PKV_F32,
                               None, 0, None, None) == b.PKV_ERR_UNSUPPORTED
    assert L.attn_decode_paged(p, p, p, p, p, p, p, 1, 1, 1, 48, 3, 64, 16, 1.0, 1, b.PKV_F32,
                               None, 0, None, None) == b.PKV_ERR_UNSUPPORTED
    assert L.attn_prefill_causal(p, p, p, p, p, 1, 16, 8, 8, 64, 1.0, b.PKV_BF16, None,
                                 None) == b.PKV_ERR_UNSUPPORTED
    # workspace needed but missing
    assert L.attn_decode_paged(p, p, p, p, p, p, p, 1, 64, 64, 8, 8, 64, 16, 1.0, 4, b.PKV_F32,
                               None, 0, None, None) == b.PKV_ERR_WORKSPACE
    # misaligned page pool
    q = ctypes.c_void_p((1 << 20) + 4)
    assert L.attn_decode_paged(p, q, p, p, p, p, p, 1, 1, 1, 8, 8, 64, 16, 1.0, 1, b.PKV_F32,
                               None, 0, None, None) == b.PKV_ERR_INVALID_ARG


def test_planner_gives_small_problems_one_split(b):
    # 1 MiB of K/V: one split and no merge launch beats 16 one-page splits plus a merge
    assert b.decode_num_splits(1, 16, 8, 8, 64, 16, 0, b.PKV_F32) == 1
    # the Llama-7B batch still splits (it fills the GPU in a few waves)
    assert b.decode_num_splits(16, 256, 32, 32, 128, 16, 0, b.PKV_BF16) > 1


def test_fp8_arguments_rejected_before_launch(b):
    L = b.lib
    p = ctypes.c_void_p(1 << 20)
    # missing scales
    assert L.attn_decode_paged_fp8(p, p, p, None, p, p, p, p, None, 1, 4, 8, 8, 8, 128, 16, 0.1, 1,
                                   None, 0, None, None) == b.PKV_ERR_INVALID_ARG
    # an odd number of KV heads: the FP8 kernel takes two per CTA
    assert L.attn_decode_paged_fp8(p, p, p, p, p, p, p, p, None, 1, 4, 8, 3, 3, 128, 16, 0.1, 1,
                                   None, 0, None, None) == b.PKV_ERR_UNSUPPORTED
    assert b.lib.attn_decode_num_splits(1, 4, 3, 3, 128, 16, 0, b.PKV_FP8_E4M3) == b.PKV_ERR_UNSUPPORTED
    # head_dim 96 is not built
    assert L.attn_decode_paged_fp8(p, p, p, p, p, p, p, p, None, 1, 4, 8, 8, 8, 96, 16, 0.1, 1,
                                   None, 0, None, None) == b.PKV_ERR_UNSUPPORTED
    # the FP8 workspace query matches the bf16 one (same fp32 partials)
    assert b.decode_workspace_size(4, 64, 32, 8, 128, 16, 8, b.PKV_FP8_E4M3) == \
        b.decode_workspace_size(4, 64, 32, 8, 128, 16, 8, b.PKV_BF16)


def test_chunked_prefill_arguments_rejected_before_launch(b):
    L = b.lib
    p = ctypes.c_void_p(1 << 20)
    args = lambda **kw: dict(dict(batch=1, chunk=8, max_blocks=4, pages=16, hq=8, hkv=8, d=128, ps=16,
                                  dtype=b.PKV_BF16, prefix=p), **kw)

    def call(**kw):
        a = args(**kw)
        return L.attn_prefill_paged_chunk(p, p, p, p, a["prefix"], p, None, a["batch"], a["chunk"],
                                          a["max_blocks"], a["pages"], a["hq"], a["hkv"], a["d"],
                                          a["ps"], 0.1, a["dtype"], None, None)

    assert call(batch=0) == b.PKV_OK                      # nothing to do
    assert call(chunk=0) == b.PKV_OK
    assert call(prefix=None) == b.PKV_ERR_INVALID_ARG      # no prefix lengths
    assert call(chunk=65) == b.PKV_ERR_INVALID_ARG         # more new tokens than the table holds
    assert call(hq=6, hkv=4) == b.PKV_ERR_INVALID_ARG      # heads not a multiple
    assert call(dtype=7) == b.PKV_ERR_INVALID_ARG
    assert call(d=64) == b.PKV_ERR_UNSUPPORTED             # only head_dim 128 is built
    assert call(ps=32, max_blocks=2) == b.PKV_ERR_UNSUPPORTED
    assert call(hq=12, hkv=4) == b.PKV_ERR_UNSUPPORTED     # a group of 3 does not divide 128 rows
    assert call(dtype=b.PKV_F32) == b.PKV_ERR_UNSUPPORTED


def test_flat_gemm_arguments_rejected_before_launch(b):
    L = b.lib
    p = ctypes.c_void_p(1 << 20)

    def call(x=p, w=p, y=p, m=8, n=4096, k=4096, dtype=b.PKV_BF16):
        return L.attn_flat_gemm(x, w, y, m, n, k, dtype, None, None)

    assert call(m=0) == b.PKV_OK                          # nothing to do
    assert call(n=0) == b.PKV_OK
    assert call(m=-1) == b.PKV_ERR_INVALID_ARG
    assert call(k=0) == b.PKV_ERR_INVALID_ARG
    assert call(x=None) == b.PKV_ERR_INVALID_ARG
    assert call(y=None) == b.PKV_ERR_INVALID_ARG
    assert call(w=ctypes.c_void_p((1 << 20) + 2)) == b.PKV_ERR_INVALID_ARG  # not 16-byte aligned
    assert call(dtype=9) == b.PKV_ERR_INVALID_ARG
    assert call(dtype=b.PKV_F32) == b.PKV_ERR_UNSUPPORTED  # bf16 only
    assert call(m=65) == b.PKV_ERR_UNSUPPORTED             # flat: at most 64 tokens
    assert call(k=100) == b.PKV_ERR_UNSUPPORTED            # rows must be 16-byte multiples


def test_flat_gemm_cluster_planning(b):
    # the split count is a cluster size: 1..8, never more CTAs than 64-column slices of K
    for m, n, k in [(1, 4096, 4096), (16, 12288, 4096), (64, 128, 64), (8, 1000, 512), (5, 70000, 64)]:
        s = b.flat_gemm_num_splits(m, n, k)
        assert 1 <= s <= 8 and s <= (k + 63) // 64
    assert b.flat_gemm_num_splits(1, 128, 64) == 1          # one slice of K
    assert b.flat_gemm_num_splits(16, 4096, 4096) == 8      # 32 tiles: the widest cluster
    assert b.lib.attn_flat_gemm_num_splits(65, 128, 64) == b.PKV_ERR_UNSUPPORTED
    assert b.lib.attn_flat_gemm_num_splits(0, 128, 64) == b.PKV_ERR_INVALID_ARG
