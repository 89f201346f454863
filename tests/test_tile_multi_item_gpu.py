"""GPU parity of the tensor-core tile kernel when its grid holds more work items than
the GPU has SMs, compared with the fp64 oracle on every output row.

One CTA of the tile kernel fills an SM, so a grid with more items than SMs makes the
running CTAs take the pending items (work stealing through cluster launch control),
and the item order (groups of (b, h), a longest-first tail) decides which CTA runs
what. Every full-size prefill launch takes that path; these tests cover it for all
three modes of the kernel: causal prefill, chunked prefill over the paged cache, and
the cascade's shared prefix. The method is tiled FlashAttention ("快速注意力内核与算子融合",
Q&A on FlashAttention tiling and on paged attention); the bf16 tolerance is the one
the other parity tests use.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_28_gb300 import workloads
from tests._compare import assert_close

pytestmark = pytest.mark.gpu

BM = 128  # query rows per tile; an item is a pair of tiles


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_28_gb300 import build
    build.build(quiet=True)
    from paged_kv_attention_28_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _prefill(b, case):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = b.prefill_causal(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _prefill_items(B, T, Hq):
    n_qt = (T + BM - 1) // BM
    return (n_qt + 1) // 2 * Hq * B


def test_causal_prefill_llama7b_all_rows(b, sms):
    """The full causal prefill workload (8 x 1024, 32/32 heads, 1024 items) on all rows."""
    case = workloads.causal_prefill_llama7b()
    assert _prefill_items(case.batch, case.seq_len, case.n_qo_heads) > 4 * sms
    out, lse = _prefill(b, case)
    wo, wl = oracle.prefill_causal(case.q.double().numpy(), case.k.double().numpy(),
                                   case.v.double().numpy(), case.scale)
    assert_close(out, wo, "bf16", "llama7b prefill out (all rows)")
    assert_close(lse, wl, "bf16", "llama7b prefill lse (all rows)")


@pytest.mark.parametrize("B,T,Hq,Hkv", [(2, 2048, 32, 8), (3, 1000, 40, 40)])
def test_causal_prefill_gqa_and_ragged_all_rows(b, sms, B, T, Hq, Hkv):
    """GQA (4 query heads per KV head) and a ragged length over more items than SMs."""
    assert _prefill_items(B, T, Hq) > sms
    case = workloads.make_prefill(300 + T + Hq, B, T, Hq, Hkv, 128, dtype="bf16")
    out, lse = _prefill(b, case)
    wo, wl = oracle.prefill_causal(case.q.double().numpy(), case.k.double().numpy(),
                                   case.v.double().numpy(), case.scale)
    assert_close(out, wo, "bf16", f"prefill B={B} T={T} {Hq}/{Hkv} out")
    assert_close(lse, wl, "bf16", f"prefill B={B} T={T} {Hq}/{Hkv} lse")


def _chunk_case(seed, n_seq, C, Hq, Hkv, prefix):
    c = workloads.make_paged_decode(seed, n_seq, Hq, Hkv, 128, 16, [p + C for p in prefix], dtype="bf16")
    gen = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((n_seq, C, Hq, 128), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return c, q, torch.tensor(prefix, dtype=torch.int32)


def _chunk(b, c, q, pl):
    d = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=d)
    out, lse = b.prefill_paged_chunk(q.to(d), c.k_pages.to(d), c.v_pages.to(d), c.block_table.to(d),
                                     pl.to(d), c.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _chunk_items(n_seq, C, Hq, Hkv):
    tpt = BM // (Hq // Hkv)
    n_qt = (C + tpt - 1) // tpt
    return (n_qt + 1) // 2 * Hkv * n_seq


@pytest.mark.parametrize("Hq,Hkv", [(32, 32), (32, 8)])
def test_chunked_prefill_many_items_all_rows(b, sms, Hq, Hkv):
    """8 sequences x 512 new tokens after prefixes of 700-1500 tokens (512 items)."""
    n_seq, C = 8, 512
    g = np.random.default_rng(Hq + Hkv)
    prefix = [int(x) for x in g.integers(700, 1501, n_seq)]
    assert _chunk_items(n_seq, C, Hq, Hkv) > sms
    c, q, pl = _chunk_case(400 + Hkv, n_seq, C, Hq, Hkv, prefix)
    out, lse = _chunk(b, c, q, pl)
    wo, wl = oracle.prefill_paged_chunk(q.double().numpy(), c.k_pages.float().numpy(),
                                        c.v_pages.float().numpy(), c.block_table.numpy(), pl.numpy(),
                                        c.scale)
    assert_close(out, wo, "bf16", f"chunk {Hq}/{Hkv} out (all rows)")
    assert_close(lse, wl, "bf16", f"chunk {Hq}/{Hkv} lse (all rows)")


def test_chunked_prefill_bench_workload_sampled_rows(b, sms):
    """The benchmarked chunk (8 sequences x 1024 new tokens after 3072, 32/32 heads, 1024
    items): about 120 sampled new tokens, every head, each checked against the oracle's decode
    over that token's visible keys (a one-token chunk is a decode of length L0 + i + 1)."""
    n_seq, C, L0, H = 8, 1024, 3072, 32
    assert _chunk_items(n_seq, C, H, H) > 4 * sms
    c, q, pl = _chunk_case(1006, n_seq, C, H, H, [L0] * n_seq)
    out, lse = _chunk(b, c, q, pl)
    g = np.random.default_rng(11)
    picks = [(int(s), int(i)) for s, i in zip(g.integers(0, n_seq, 96), g.integers(0, C, 96))]
    picks += [(0, 0), (7, C - 1), (3, 127), (3, 128), (5, 511), (5, 512)] + [(s, C - 1) for s in range(n_seq)]
    picks += [(s, 0) for s in range(n_seq)] + [(1, 255), (2, 256)]
    seqs = np.array([s for s, _ in picks])
    toks = np.array([i for _, i in picks])
    qd = q.double().numpy()[seqs, toks]                                  # [N, H, D]
    wo, wl = oracle.decode_paged(qd, c.k_pages.float().numpy(), c.v_pages.float().numpy(),
                                 c.block_table.numpy()[seqs], L0 + toks + 1, c.scale)
    assert_close(out[seqs, toks], wo, "bf16", "chunk bench workload sampled out")
    assert_close(lse[seqs, :, toks], wl, "bf16", "chunk bench workload sampled lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("R,prefix,Hq,Hkv", [(640, 512, 64, 8), (1280, 384, 32, 8)])
def test_cascade_prefix_many_items_all_rows(b, sms, R, prefix, Hq, Hkv):
    """More (KV head, row pair) prefix items than SMs: 160 of them, one prefix chunk each."""
    G = Hq // Hkv
    items = Hkv * ((R * G + 2 * BM - 1) // (2 * BM))
    assert items > sms
    c = workloads.make_cascade(500 + R, R, prefix, (0, 40), Hq, Hkv, 128, page_size=16, dtype="bf16")
    d = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=d)
    out, lse = b.decode_cascade(c.q.to(d), c.k_pages.to(d), c.v_pages.to(d), c.prefix_table.to(d),
                                c.prefix_len, c.suffix_table.to(d), c.suffix_lens.to(d), c.scale,
                                err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wo, wl = oracle.cascade_decode(c.q.double().numpy(), c.k_pages.float().numpy(),
                                   c.v_pages.float().numpy(), c.prefix_table.numpy(), c.prefix_len,
                                   c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)
    assert_close(out.float().cpu().numpy(), wo, "bf16", f"cascade R={R} out (all rows)")
    assert_close(lse.cpu().numpy(), wl, "bf16", f"cascade R={R} lse (all rows)")
