"""GPU parity of attn_flat_gemm (tcgen05 flat GEMM, K split over a cluster) against the fp64
oracle ``Y = X W^T`` on the same seeded bf16 inputs, every output element compared.

The shapes cover one token (the GEMV case), the page's padded sizes (8, 16) and token
counts that pad to 32 and 64, a ragged n and ragged k, a single CTA per tile and
clusters of 2 to 8 CTAs, and the Llama-2-7B-shaped QKV and O projections at full size
("【FlashAttention-V4，非官方】FlashDecoding++", sections 1, 2 and 4). The tolerance is the
bf16 bar of the other parity tests.
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
    return binding


def run(b, case):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = b.flat_gemm(case.x.cuda(), case.w.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return y.float().cpu().numpy()


@pytest.mark.parametrize("m,n,k", [
    (1, 128, 64),       # one slice of K: one CTA per tile, no cluster
    (3, 200, 72),       # ragged n (a partial tile) and ragged k (a partial slice)
    (8, 1000, 512),     # the page's padded token count
    (16, 384, 4096),    # three tiles, a cluster of 8 splitting K
    (17, 640, 1000),    # pads to 32 tokens; k not a multiple of 64
    (40, 256, 2048),    # pads to 64 tokens
    (64, 1536, 4096),   # the largest token count built
    (5, 70000, 64),     # more tiles than resident CTAs
])
def test_flat_gemm_matches_oracle(b, m, n, k):
    case = workloads.make_flat_gemm(700 + m + n % 97, m, n, k)
    y = run(b, case)
    want = oracle.flat_gemm(case.x.double().numpy(), case.w.double().numpy())
    assert_close(y, want, "bf16", f"flat gemm {m}x{n}x{k}")


@pytest.mark.parametrize("m", [1, 8, 16])
@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_flat_gemm_llama7b_projections(b, proj, m):
    case = (workloads.llama7b_qkv_projection if proj == "qkv" else workloads.llama7b_o_projection)(m)
    assert b.flat_gemm_num_splits(m, case.n, case.k) > 1
    y = run(b, case)
    want = oracle.flat_gemm(case.x.double().numpy(), case.w.double().numpy())
    assert_close(y, want, "bf16", f"{case.name}")


def test_flat_gemm_repeated_calls_agree(b):
    """The cluster sums its partial tiles in rank order: two calls give identical bits."""
    case = workloads.llama7b_o_projection(16)
    y1 = run(b, case)
    y2 = run(b, case)
    assert np.array_equal(y1, y2)
