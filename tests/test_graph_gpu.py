"""The entry points inside a captured CUDA graph.

Every call only enqueues work on the given stream (no allocation, no synchronisation), so a
training or serving loop can capture forward, backward and decoding once and replay them. The
captured kernels keep the arguments of the capture (device pointers, tensor maps encoded then),
so each replay here first copies new inputs into the captured buffers and the results must match
eager calls on the same inputs: bit for bit where the kernels are deterministic (O, lse, dK, dV,
decoding), within fp32 reduction-order rounding for dQ.
"""
import pytest
import torch

from exact_attention_fa_gb300 import binding as fa

pytestmark = pytest.mark.gpu


def _bf16(shape, g, device):
    return torch.randn(shape, generator=g, device="cpu").to(device=device, dtype=torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_forward_backward_graph_replay(cuda, d):
    B, Hh, N = 2, 4, 640
    scale = d ** -0.5
    g = torch.Generator().manual_seed(81)
    q, k, v, do = (_bf16((B, Hh, N, d), g, cuda) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, N), dtype=torch.float32, device=cuda)
    dq = torch.empty((B, Hh, N, d), dtype=torch.float32, device=cuda)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, Hh, N, d), dtype=torch.uint8, device=cuda)

    # warm-up on a side stream (the library's per-device set-up happens outside the capture)
    s = torch.cuda.Stream(cuda)
    s.wait_stream(torch.cuda.current_stream(cuda))
    with torch.cuda.stream(s):
        fa.fa_fwd(q, k, v, o, lse, scale, True)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, True, ws)
    torch.cuda.current_stream(cuda).wait_stream(s)
    torch.cuda.synchronize(cuda)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_fwd(q, k, v, o, lse, scale, True)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, True, ws)

    for step in range(3):
        for t in (q, k, v, do):
            t.copy_(_bf16(t.shape, g, cuda))
        graph.replay()
        torch.cuda.synchronize(cuda)
        fa.fa_check_device_error()
        o_ref, lse_ref = fa.attention_forward(q, k, v, scale, causal=True)
        dq_ref, dk_ref, dv_ref = fa.attention_backward(q, k, v, o_ref, lse_ref, do, scale,
                                                       causal=True)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), step
        assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref), step
        err = (torch.linalg.vector_norm(dq - dq_ref) / torch.linalg.vector_norm(dq_ref)).item()
        assert err <= 1e-5, (step, err)


@pytest.mark.parametrize("nq,d", [(1, 128), (8, 64)])
def test_decode_graph_replay(cuda, nq, d):
    """Decoding is two kernels, the merge launched as a programmatic dependent of the split
    kernel; captured, that dependency is an edge of the graph."""
    B, Hh, Nk = 2, 8, 3000
    scale = d ** -0.5
    g = torch.Generator().manual_seed(82)
    q = _bf16((B, Hh, nq, d), g, cuda)
    k, v = (_bf16((B, Hh, Nk, d), g, cuda) for _ in range(2))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, nq), dtype=torch.float32, device=cuda)
    ws = torch.empty(fa.fa_decode_workspace_bytes(B, Hh, nq, Nk, d), dtype=torch.uint8,
                     device=cuda)
    s = torch.cuda.Stream(cuda)
    s.wait_stream(torch.cuda.current_stream(cuda))
    with torch.cuda.stream(s):
        fa.fa_decode(q, k, v, o, lse, scale, 0, ws)
    torch.cuda.current_stream(cuda).wait_stream(s)
    torch.cuda.synchronize(cuda)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_decode(q, k, v, o, lse, scale, 0, ws)

    for step in range(3):
        for t in (q, k, v):
            t.copy_(_bf16(t.shape, g, cuda))
        graph.replay()
        torch.cuda.synchronize(cuda)
        fa.fa_check_device_error()
        o_ref, lse_ref = fa.attention_decode(q, k, v, scale)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), step
