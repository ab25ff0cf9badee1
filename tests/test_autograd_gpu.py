"""The autograd wrapper: gradients that flow through `attention` are the library's backward.

Compared with the explicit calls on the same inputs (dK, dV bit for bit; dQ, an fp32 reduction
returned in bf16, within a bf16 rounding) and, for every head, with the oracle's gradients at the
backward's bound (relative Frobenius 2e-2).
"""
import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl
from oracle import attention as orc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal,sparse", [(True, False), (False, True), (True, True)])
def test_autograd_matches_backward_and_oracle(cuda, causal, sparse):
    w = wl.Workload("autograd", 1, 2, 300, 64, causal=causal, block_sparse=sparse, seed=78)
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, cuda) for n in ("q", "k", "v", "do"))
    mask_np = inp.raw("mask") if sparse else None
    mask = torch.from_numpy(mask_np).to(cuda) if sparse else None
    ql, kl, vl = (t.clone().requires_grad_(True) for t in (q, k, v))
    o, lse = fa.attention(ql, kl, vl, causal=causal, block_mask=mask)
    (o.float() * do.float()).sum().backward()
    fa.fa_check_device_error()

    o_ref, lse_ref = fa.attention_forward(q, k, v, causal=causal, block_mask=mask)
    dq, dk, dv = fa.attention_backward(q, k, v, o_ref, lse_ref, do, causal=causal,
                                       block_mask=mask)
    assert torch.equal(o.detach(), o_ref) and torch.equal(lse, lse_ref)
    assert torch.equal(kl.grad, dk) and torch.equal(vl.grad, dv)
    assert ql.grad.dtype == torch.bfloat16
    assert (ql.grad.float() - dq).abs().max().item() <= 2 ** -7 * dq.abs().max().item()

    for h in range(w.H):
        qf, kf, vf, dof = (inp.f64_head(n, 0, h) for n in ("q", "k", "v", "do"))
        gq, gk, gv = orc.backward_head(qf, kf, vf, dof, w.softmax_scale, causal=causal,
                                       block_mask=mask_np)
        for got, want in ((ql.grad, gq), (kl.grad, gk), (vl.grad, gv)):
            err = H.rel_fro(got[0, h].float().cpu().numpy(), want)
            assert err <= H.GRAD_REL_FRO, (h, err)


def test_autograd_rejects_non_bf16(cuda):
    q = torch.zeros(1, 1, 16, 64, device=cuda)
    with pytest.raises(ValueError):
        fa.attention(q, q, q)
