"""CUDA-graph capture of the library's calls.

No call allocates device memory, copies to the host or synchronises, so each one can be
captured into a CUDA graph once and replayed. A replay reads the current contents of the
captured buffers: the tests write new inputs into the same buffers, replay, and check the
result against the fp64 oracle (or, for the cascade, against a direct call on the same
inputs, which launches the same kernels).
"""
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


def capture(fn):
    """One warm-up call on a side stream (one-time kernel attributes and library state),
    then the capture of a second call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def new_q(shape, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


@pytest.mark.parametrize("which,splits,phi", [("single_seq_decode_f32", 4, None),
                                              ("gqa_small", 8, None), ("gqa_small", 8, 0.0)])
def test_decode_graph_replays_on_new_queries(b, which, splits, phi):
    if which == "single_seq_decode_f32":
        c = workloads.single_seq_decode_f32()
    else:
        c = workloads.make_paged_decode(4242, 3, 16, 4, 128, 16, [700, 33, 1500], num_pages=256,
                                        dtype="bf16")
    d = "cuda"
    q, kp, vp, bt, ln = (t.to(d) for t in (c.q, c.k_pages, c.v_pages, c.block_table, c.kv_lens))
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=d)
    ws = b.alloc_workspace(b.decode_workspace_size(c.batch, c.max_blocks, c.n_qo_heads, c.n_kv_heads,
                                                   c.head_dim, c.page_size, splits,
                                                   b.PKV_F32 if c.dtype_name == "f32" else b.PKV_BF16), d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    fb = torch.zeros(1, dtype=torch.int32, device=d)

    def call():
        b.decode_paged(q, kp, vp, bt, ln, c.scale, num_splits=splits, out=out, lse=lse, workspace=ws,
                       err_flag=err, unified_phi=phi, fallback_count=fb if phi is not None else None)

    g = capture(call)
    for seed in (11, 12):
        qn = new_q(tuple(c.q.shape), c.q.dtype, seed)
        q.copy_(qn)
        g.replay()
        torch.cuda.synchronize()
        want = oracle.decode_paged(qn.double().numpy(), c.k_pages.float().numpy(),
                                   c.v_pages.float().numpy(), c.block_table.numpy(),
                                   c.kv_lens.numpy(), c.scale)
        assert_close(out.float().cpu().numpy(), want[0], c.dtype_name, f"{which} replay out")
        assert_close(lse.cpu().numpy(), want[1], c.dtype_name, f"{which} replay lse")
    assert int(err.item()) == 0


def test_prefill_graph_replays_on_new_queries(b):
    c = workloads.make_prefill(77, 1, 300, 2, 2, 128, dtype="bf16")
    d = "cuda"
    q, k, v = c.q.to(d), c.k.to(d), c.v.to(d)
    out = torch.empty_like(q)
    lse = torch.empty((c.batch, c.n_qo_heads, c.seq_len), dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    g = capture(lambda: b.prefill_causal(q, k, v, c.scale, out=out, lse=lse, err_flag=err))
    qn = new_q(tuple(c.q.shape), c.q.dtype, 13)
    q.copy_(qn)
    g.replay()
    torch.cuda.synchronize()
    wo, wl = oracle.prefill_causal(qn.double().numpy(), c.k.double().numpy(), c.v.double().numpy(),
                                   c.scale)
    assert_close(out.float().cpu().numpy(), wo, "bf16", "prefill replay out")
    assert_close(lse.cpu().numpy(), wl, "bf16", "prefill replay lse")
    assert int(err.item()) == 0


def test_cascade_graph_replay_matches_direct_call(b):
    # The cascade call forks its prefix kernel onto the library's side stream and joins it
    # back with events; the capture records that fork and join as graph edges.
    c = workloads.make_cascade(88, 12, 1008, [40, 300, 17, 129, 64, 500, 1, 256, 255, 90, 77, 400],
                               16, 4, 128, page_size=16, dtype="bf16")
    d = "cuda"
    q, kp, vp, pt, st, sl = (t.to(d) for t in (c.q, c.k_pages, c.v_pages, c.prefix_table,
                                               c.suffix_table, c.suffix_lens))
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=d)
    ws = b.alloc_workspace(b.cascade_workspace_size(c.n_requests, c.prefix_len, st.shape[1],
                                                    c.n_qo_heads, c.n_kv_heads, c.head_dim,
                                                    c.page_size), d)
    err = torch.zeros(1, dtype=torch.int32, device=d)

    def call(o, l):
        b.decode_cascade(q, kp, vp, pt, c.prefix_len, st, sl, c.scale, out=o, lse=l, workspace=ws,
                         err_flag=err)

    g = capture(lambda: call(out, lse))
    qn = new_q(tuple(c.q.shape), c.q.dtype, 14)
    q.copy_(qn)
    g.replay()
    torch.cuda.synchronize()
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    call(out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    want = oracle.cascade_decode(qn.double().numpy(), c.k_pages.float().numpy(),
                                 c.v_pages.float().numpy(), c.prefix_table.numpy(), c.prefix_len,
                                 c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)
    assert_close(out.float().cpu().numpy(), want[0], "bf16", "cascade replay out")
    assert_close(lse.cpu().numpy(), want[1], "bf16", "cascade replay lse")
    assert int(err.item()) == 0
