"""GPU parity of attn_prefill_paged_chunk (chunked prefill over the paged cache, on the
tensor cores) against the fp64 oracle on the same seeded inputs.

The pools come from the decode workload builder with the full length prefix + chunk of
every sequence, so unused pages and the slots past each sequence's end hold NaN: the
kernel must neither read them into a result nor let them reach PV."""
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


def make(seed, C, Hq, Hkv, prefix):
    prefix = list(prefix)
    c = workloads.make_paged_decode(seed, len(prefix), Hq, Hkv, 128, 16, [p + C for p in prefix],
                                    dtype="bf16")
    gen = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((len(prefix), C, Hq, 128), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return c, q, torch.tensor(prefix, dtype=torch.int32)


@pytest.mark.parametrize("C,Hq,Hkv,prefix", [
    (100, 8, 2, (0, 300)),          # G = 4, one sequence with no prefix
    (300, 2, 2, (1000,)),           # G = 1, three query tiles, prefix not page aligned
    (1, 16, 2, (5, 0, 130)),        # a one-token chunk (decode through the prefill path), G = 8
    (257, 4, 2, (17, 127)),         # G = 2, ragged chunk, prefixes straddling tile edges
])
def test_prefill_paged_chunk_matches_oracle(b, C, Hq, Hkv, prefix):
    c, q, pl = make(90 + C + Hq, C, Hq, Hkv, prefix)
    d = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=d)
    out, lse = b.prefill_paged_chunk(q.to(d), c.k_pages.to(d), c.v_pages.to(d), c.block_table.to(d),
                                     pl.to(d), c.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wo, wl = oracle.prefill_paged_chunk(q.double().numpy(), c.k_pages.float().numpy(),
                                        c.v_pages.float().numpy(), c.block_table.numpy(), pl.numpy(),
                                        c.scale)
    assert_close(out.float().cpu().numpy(), wo, "bf16", f"chunk C={C} G={Hq // Hkv} out")
    assert_close(lse.cpu().numpy(), wl, "bf16", f"chunk C={C} G={Hq // Hkv} lse")


def test_prefill_paged_chunk_bad_page_sets_flag(b):
    c, q, pl = make(95, 40, 4, 2, (20, 20))
    table = c.block_table.clone()
    table[1, 0] = c.num_pages + 3                   # inside sequence 1
    d = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=d)
    b.prefill_paged_chunk(q.to(d), c.k_pages.to(d), c.v_pages.to(d), table.to(d), pl.to(d), c.scale,
                          err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & b.PKV_DEVERR_BAD_PAGE
