"""GPU parity on seeded random shapes: the decode (both kernels), the causal prefill and the
chunked prefill, each compared with the fp64 oracle on every output row and LSE.

The shapes are drawn from a fixed seed, so every run checks the same cases: lengths that
fall on and off page and tile edges, empty sequences, GQA groups of 1 to 8, head_dim 64 and
128, split counts from the planner's choice up to 32, and pools whose unused page slots are
poisoned with non-finite values."""
import random

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


def _decode_cases(n, seed):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        dt = rng.choice(["f32", "bf16", "bf16"])
        D = 128 if dt == "bf16" and rng.random() < 0.7 else rng.choice([64, 128])
        G = rng.choice([1, 2, 4, 8])
        Hkv = rng.choice([1, 2, 4, 8])
        Bn = rng.choice([1, 2, 3, 5])
        lens = [rng.choice([0, 1, 15, 16, 17, 100, 255, 256, 700, 1500]) for _ in range(Bn)]
        if max(lens) == 0:
            lens[0] = 300
        S = rng.choice([0, 0, 1, 2, 3, 7, 32])
        cases.append((i, dt, D, G, Hkv, Bn, tuple(lens), S, rng.randrange(1 << 20), rng.choice([1.0, 2.0])))
    return cases


@pytest.mark.parametrize("i,dt,D,G,Hkv,Bn,lens,S,seed,k_std", _decode_cases(24, 2024))
def test_decode_random_shape(b, i, dt, D, G, Hkv, Bn, lens, S, seed, k_std):
    c = workloads.make_paged_decode(seed, Bn, G * Hkv, Hkv, D, page_size=16, kv_lens=list(lens), dtype=dt,
                                    poison=True, k_std=k_std, name=f"random_decode_{i}")
    dev = torch.device("cuda")
    q, kp, vp, bt, ln = (t.to(dev) for t in (c.q, c.k_pages, c.v_pages, c.block_table, c.kv_lens))
    tdt = b.PKV_F32 if dt == "f32" else b.PKV_BF16
    ws = b.alloc_workspace(b.decode_workspace_size(Bn, c.max_blocks, G * Hkv, Hkv, D, 16, S, tdt), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = b.decode_paged(q, kp, vp, bt, ln, c.scale, num_splits=S, workspace=ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wo, wl = oracle.decode_paged(c.q.double().numpy(), c.k_pages.float().numpy(), c.v_pages.float().numpy(),
                                 c.block_table.numpy(), c.kv_lens.numpy(), c.scale)
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    empty = np.array(lens) == 0
    assert np.all(o[empty] == 0) and np.all(np.isneginf(l[empty]))
    assert_close(o[~empty], wo[~empty], dt, f"decode case {i} out")
    assert_close(l[~empty], wl[~empty], dt, f"decode case {i} lse")


def _prefill_cases(n, seed):
    rng = random.Random(seed)
    return [(i, rng.choice([1, 2]), rng.choice([1, 63, 127, 128, 129, 200, 255, 384, 513, 640]),
             rng.choice([1, 2, 4]), rng.choice([1, 2, 3]), rng.randrange(1 << 20)) for i in range(n)]


@pytest.mark.parametrize("i,Bn,T,G,Hkv,seed", _prefill_cases(10, 2025))
def test_prefill_random_shape(b, i, Bn, T, G, Hkv, seed):
    case = workloads.make_prefill(seed, Bn, T, G * Hkv, Hkv, 128, dtype="bf16")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = b.prefill_causal(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wo, wl = oracle.prefill_causal(case.q.double().numpy(), case.k.double().numpy(), case.v.double().numpy(),
                                   case.scale)
    assert_close(out.float().cpu().numpy(), wo, "bf16", f"prefill case {i} out")
    assert_close(lse.cpu().numpy(), wl, "bf16", f"prefill case {i} lse")


def _chunk_cases(n, seed):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        Bn = rng.choice([1, 2, 3])
        cases.append((i, rng.choice([1, 2, 4, 8]), rng.choice([1, 2]), Bn, rng.choice([16, 33, 100, 128, 200]),
                      tuple(rng.choice([0, 5, 16, 100, 300]) for _ in range(Bn)), rng.randrange(1 << 20)))
    return cases


@pytest.mark.parametrize("i,G,Hkv,Bn,C,pre,seed", _chunk_cases(8, 2026))
def test_chunked_prefill_random_shape(b, i, G, Hkv, Bn, C, pre, seed):
    Hq = G * Hkv
    c = workloads.make_paged_decode(seed, Bn, Hq, Hkv, 128, page_size=16, kv_lens=[p + C for p in pre],
                                    dtype="bf16", poison=True, name=f"random_chunk_{i}")
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    qc = torch.randn(Bn, C, Hq, 128, generator=g).to(torch.bfloat16)
    pl = torch.tensor(pre, dtype=torch.int32)
    dev = torch.device("cuda")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = b.prefill_paged_chunk(qc.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
                                     pl.to(dev), c.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wo, wl = oracle.prefill_paged_chunk(qc.double().numpy(), c.k_pages.float().numpy(), c.v_pages.float().numpy(),
                                        c.block_table.numpy(), pl.numpy(), c.scale)
    assert_close(out.float().cpu().numpy(), wo, "bf16", f"chunk case {i} out")
    assert_close(lse.cpu().numpy(), wl, "bf16", f"chunk case {i} lse")
