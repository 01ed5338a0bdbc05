"""CUDA-graph capture of the library's calls (a serving loop replays a captured
step): a replay must run the same kernels as a direct call, read the inputs'
current contents, and give bit-identical results.  Covers the single-tile and
two-tile forward, the split-KV forward with its programmatic dependent merge
launch, and the backward."""
import pytest

torch = pytest.importorskip("torch")

import exact_attention_19_gb300 as fa  # noqa: E402

pytestmark = pytest.mark.gpu


def _rand(shape, gen):
    return torch.randn(shape, device="cuda", dtype=torch.bfloat16, generator=gen)


@pytest.mark.parametrize("B,H,N,d,causal,split", [
    (2, 4, 1024, 64, True, False),    # one query tile per CTA, two CTAs per SM
    (1, 4, 1000, 128, True, False),   # two query tiles per CTA
    (1, 1, 4096, 64, False, True),    # split-KV: sliced forward + merge (programmatic dependent launch)
    (2, 40, 1000, 128, False, False),  # persistent kernel, static schedule, more units than SMs
    (4, 12, 512, 64, False, False),    # persistent kernel at d = 64 (two Q buffers per tile)
    (4, 64, 2200, 64, True, False),    # persistent kernel under cluster launch control
    (16, 48, 1100, 128, True, False),  # the same at d = 128 (20+ query-tile pairs per SM)
])
def test_forward_graph_replay_matches_direct_calls(B, H, N, d, causal, split):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + N + d)
    q, k, v = (_rand((B, H, N, d), gen) for _ in range(3))
    n_splits = fa.fa_splitkv_heuristic(B, H, N, N, d, int(causal)) if split else 1
    if split:
        assert n_splits > 1
    ws = (torch.empty(fa.fa_splitkv_workspace_bytes(B, H, N, N, d, n_splits), dtype=torch.uint8, device="cuda")
          if n_splits > 1 else None)
    o_g, lse_g = torch.empty_like(q), torch.empty(B, H, N, device="cuda")

    def step(o, lse):
        fa.fwd(q, k, v, causal=causal, out=o, lse=lse, n_splits=n_splits, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step(o_g, lse_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(o_g, lse_g)
    for round_ in range(2):
        if round_ == 1:  # new input values in place: the replay must read them
            for t in (q, k, v):
                t.copy_(_rand(t.shape, gen))
        o_d, lse_d = torch.empty_like(q), torch.empty(B, H, N, device="cuda")
        step(o_d, lse_d)
        o_g.zero_()
        lse_g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_d), f"O differs after replay {round_}"
        assert torch.equal(lse_g, lse_d), f"LSE differs after replay {round_}"
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, hex(word)


def test_backward_graph_replay_matches_direct_calls():
    B, H, N, d, causal = 2, 3, 700, 128, True
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    q, k, v, do = (_rand((B, H, N, d), gen) for _ in range(4))
    o, lse = fa.fwd(q, k, v, causal=causal, n_splits=1)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device="cuda")
    g_out = [torch.empty_like(q) for _ in range(3)]

    def step(outs):
        fa.bwd(q, k, v, o, lse, do, causal=causal, dq=outs[0], dk=outs[1], dv=outs[2], workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(g_out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(g_out)
    do.copy_(_rand(do.shape, gen))  # new upstream gradient in place
    d_out = [torch.empty_like(q) for _ in range(3)]
    step(d_out)
    for t in g_out:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), g_out, d_out):
        assert torch.equal(a, b), f"{name} differs after replay"
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, hex(word)
