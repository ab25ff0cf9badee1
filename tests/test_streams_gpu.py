"""Calls on several streams at once: the library keeps no per-call state outside the caller's
buffers (the backward's work counters and statistics live in its workspace, decoding's pieces in
its own), so concurrent calls on different streams give what the same calls give one after the
other -- bit for bit where the kernels are deterministic (O, lse, dK, dV, decoding), within fp32
reduction-order rounding for dQ."""
import pytest
import torch

from exact_attention_fa_gb300 import binding as fa

pytestmark = pytest.mark.gpu


def _case(g, device, B, H, N, d):
    mk = lambda: torch.randn((B, H, N, d), generator=g).to(device=device, dtype=torch.bfloat16)
    q, k, v, do = mk(), mk(), mk(), mk()
    return dict(q=q, k=k, v=v, do=do, o=torch.empty_like(q),
                lse=torch.empty((B, H, N), dtype=torch.float32, device=device),
                dq=torch.empty((B, H, N, d), dtype=torch.float32, device=device),
                dk=torch.empty_like(k), dv=torch.empty_like(v),
                ws=torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                               device=device))


def _run(c, causal):
    scale = c["q"].shape[-1] ** -0.5
    fa.fa_fwd(c["q"], c["k"], c["v"], c["o"], c["lse"], scale, causal)
    fa.fa_bwd(c["q"], c["k"], c["v"], c["o"], c["do"], c["lse"], c["dq"], c["dk"], c["dv"], scale,
              causal, c["ws"])


def test_forward_backward_on_concurrent_streams(cuda):
    g = torch.Generator().manual_seed(83)
    cases = [_case(g, cuda, 2, 4, 1536, 128), _case(g, cuda, 1, 8, 2048, 64),
             _case(g, cuda, 3, 2, 777, 128), _case(g, cuda, 2, 3, 1000, 64)]
    causal = [True, False, True, True]
    # one after the other
    want = []
    for c, cz in zip(cases, causal):
        _run(c, cz)
        torch.cuda.synchronize(cuda)
        want.append({n: c[n].clone() for n in ("o", "lse", "dq", "dk", "dv")})
        for n in ("o", "lse", "dq", "dk", "dv"):
            c[n].fill_(float("nan"))
    fa.fa_check_device_error()
    # all at once, one stream each, several rounds
    streams = [torch.cuda.Stream(cuda) for _ in cases]
    for _ in range(3):
        torch.cuda.synchronize(cuda)
        for c, cz, s in zip(cases, causal, streams):
            with torch.cuda.stream(s):
                _run(c, cz)
        torch.cuda.synchronize(cuda)
        fa.fa_check_device_error()
        for c, w in zip(cases, want):
            for n in ("o", "lse", "dk", "dv"):
                assert torch.equal(c[n], w[n]), n
            err = (torch.linalg.vector_norm(c["dq"] - w["dq"]) / torch.linalg.vector_norm(w["dq"])).item()
            assert err <= 1e-5, err


def test_decode_on_concurrent_streams(cuda):
    g = torch.Generator().manual_seed(84)
    B, H, Nk, d = 2, 8, 5000, 128
    calls = []
    for nq in (1, 4, 8):
        q = torch.randn((B, H, nq, d), generator=g).to(device=cuda, dtype=torch.bfloat16)
        k, v = (torch.randn((B, H, Nk, d), generator=g).to(device=cuda, dtype=torch.bfloat16)
                for _ in range(2))
        ws = torch.empty(fa.fa_decode_workspace_bytes(B, H, nq, Nk, d), dtype=torch.uint8,
                         device=cuda)
        calls.append((q, k, v, torch.empty_like(q),
                      torch.empty((B, H, nq), dtype=torch.float32, device=cuda), ws))
    want = []
    for q, k, v, o, lse, ws in calls:
        fa.fa_decode(q, k, v, o, lse, d ** -0.5, 0, ws)
        torch.cuda.synchronize(cuda)
        want.append((o.clone(), lse.clone()))
    streams = [torch.cuda.Stream(cuda) for _ in calls]
    for _ in range(3):
        torch.cuda.synchronize(cuda)
        for (q, k, v, o, lse, ws), s in zip(calls, streams):
            with torch.cuda.stream(s):
                o.fill_(float("nan"))
                fa.fa_decode(q, k, v, o, lse, d ** -0.5, 0, ws)
        torch.cuda.synchronize(cuda)
        fa.fa_check_device_error()
        for (q, k, v, o, lse, ws), (wo, wl) in zip(calls, want):
            assert torch.equal(o, wo) and torch.equal(lse, wl)
