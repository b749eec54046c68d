"""``fa.attention``: the autograd node over the forward and backward entry
points.  The gradients autograd returns are the backward call's, and they
match the fp64 oracle."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from oracle import attention_backward
from parity import TOL_GRAD, TOL_O, check_close, check_lse, oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_autograd_matches_the_backward_call_and_the_oracle(d, causal):
    inp = make_inputs(B=2, H=3, N=300, d=d, mask="causal" if causal else "none", seed=23 + d)
    q, k, v = (inp[x].cuda().requires_grad_(True) for x in ("q", "k", "v"))
    do = inp["do"].cuda()
    o, lse = fa.attention(q, k, v, causal=causal, return_lse=True)
    (o.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK

    # the same as calling the entry points directly (dQ is summed in any
    # order, so within rounding; the rest bit for bit)
    o2, lse2 = fa.forward(q.detach(), k.detach(), v.detach(), causal=causal)
    dq2, dk2, dv2 = fa.backward(q.detach(), k.detach(), v.detach(), o2, lse2, do, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(k.grad, dk2) and torch.equal(v.grad, dv2)
    scale_q = dq2.float().abs().max().item()
    assert (q.grad.float() - dq2.float()).abs().max().item() <= 1e-2 * scale_q

    qq, kk, vv, dd = oracle_inputs(inp)
    rdq, rdk, rdv, ro, rlse, _ = attention_backward(qq, kk, vv, dd, inp["scale"], causal=causal)
    check_close("O", o.detach().double().cpu().numpy(), ro, TOL_O)
    check_lse(lse.double().cpu().numpy(), rlse)
    for name, got, want in (("dQ", q.grad, rdq), ("dK", k.grad, rdk), ("dV", v.grad, rdv)):
        check_close(name, got.double().cpu().numpy(), want, TOL_GRAD)


def test_autograd_through_a_composite_loss():
    # attention inside a larger graph: the gradient reaching O is not dO of
    # a plain sum, and only some inputs need gradients
    inp = make_inputs(B=1, H=2, N=256, d=64, mask="causal", seed=5)
    q = inp["q"].cuda().requires_grad_(True)
    k, v = inp["k"].cuda(), inp["v"].cuda()
    w = torch.linspace(-1, 1, 64, device="cuda")
    o = fa.attention(q, k, v, causal=True)
    loss = (torch.tanh(o.float()) * w).sum()
    loss.backward()
    # reference: the same composite on the fp64 oracle
    qq, kk, vv, _ = oracle_inputs(inp)
    o64 = torch.from_numpy(np.ascontiguousarray(
        attention_backward(qq, kk, vv, np.zeros_like(qq), inp["scale"], causal=True)[3]))
    g_o = ((1 - torch.tanh(o64) ** 2) * w.double().cpu()).numpy()  # dloss/dO at the oracle's O
    rdq = attention_backward(qq, kk, vv, g_o, inp["scale"], causal=True)[0]
    check_close("dQ", q.grad.double().cpu().numpy(), rdq, TOL_GRAD)
    assert k.grad is None and v.grad is None
