"""GPU parity of attn_prefill_causal (tcgen05 kernel) against the fp64 oracle."""
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
    out, lse = b.prefill_causal(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("B,T,Hq,Hkv", [(1, 1, 1, 1), (1, 128, 2, 2), (2, 200, 2, 2), (1, 129, 4, 2),
                                        (1, 384, 4, 1), (2, 255, 2, 2), (1, 1000, 2, 2)])
def test_prefill_small_all_rows(b, B, T, Hq, Hkv):
    case = workloads.make_prefill(50 + T + Hq, B, T, Hq, Hkv, 128, dtype="bf16")
    out, lse = run(b, case)
    wo, wl = oracle.prefill_causal(case.q.double().numpy(), case.k.double().numpy(),
                                   case.v.double().numpy(), case.scale)
    assert_close(out, wo, "bf16", f"prefill T={T} out")
    assert_close(lse, wl, "bf16", f"prefill T={T} lse")


def test_prefill_wide_logits(b):
    """Larger inputs push logits far apart, so every tile moves the running max."""
    case = workloads.make_prefill(61, 1, 512, 2, 2, 128, dtype="bf16", std=2.5)
    out, lse = run(b, case)
    wo, wl = oracle.prefill_causal(case.q.double().numpy(), case.k.double().numpy(),
                                   case.v.double().numpy(), case.scale)
    assert_close(out, wo, "bf16", "wide out")
    assert_close(lse, wl, "bf16", "wide lse")


def test_causal_prefill_llama7b_sampled_rows(b):
    case = workloads.causal_prefill_llama7b()
    out, lse = run(b, case)
    g = np.random.default_rng(4)
    T = case.seq_len
    rows = [(bb, h, i) for bb, h, i in zip(g.integers(0, case.batch, 300),
                                           g.integers(0, case.n_qo_heads, 300),
                                           g.integers(0, T, 300))]
    rows += [(0, 0, 0), (7, 31, T - 1), (3, 5, 127), (3, 5, 128), (1, 9, 511), (1, 9, 512)]
    wo, wl = oracle.prefill_causal(case.q.double().numpy(), case.k.double().numpy(),
                                   case.v.double().numpy(), case.scale, rows=rows)
    idx = tuple(np.array(rows).T)
    got_o = out[idx[0], idx[2], idx[1]]
    want_o = wo[idx[0], idx[2], idx[1]]
    assert_close(got_o, want_o, "bf16", "llama7b prefill sampled out")
    assert_close(lse[idx], wl[idx], "bf16", "llama7b prefill sampled lse")
    # properties that hold at any size: row 0 of every (b, h) is v_0 (up to bf16 output rounding)
    v0 = case.v[:, 0].float().numpy()
    assert np.abs(out[:, 0] - v0).max() <= 2e-2
    assert np.isfinite(out).all() and np.isfinite(lse).all()
