"""Launch order of the backward's kernels.  fa_backward lets each kernel
after the first start while the one before it finishes (programmatic
dependent launch) and wait for that kernel's results before it reads them.
Calls queued back to back on one stream, sharing one workspace, must each
see their own preprocess (LSE, D, the cleared dQ accumulator) and their own
split plan: the results must equal those of the same calls made one at a
time with the stream drained in between.  A backward captured in a CUDA
graph keeps that order on every replay.  Marked ``gpu``."""

import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from parity import to_device

pytestmark = pytest.mark.gpu


def one_at_a_time(g, o, lse, dos, ws, kw):
    out = []
    for do in dos:
        torch.cuda.synchronize()
        r = fa.backward(g["q"], g["k"], g["v"], o, lse, do, workspace=ws, **kw)
        torch.cuda.synchronize()
        out.append(tuple(t.clone() for t in r))
    return out


@pytest.mark.parametrize("d,mask", [(64, "causal"), (128, "causal"), (64, "band_global"),
                                    (128, "none")])
def test_back_to_back_calls_see_their_own_preprocess(d, mask):
    extra = dict(global_every=4) if mask == "band_global" else {}
    inp = make_inputs(B=1, H=4, N=1536, d=d, mask=mask, seed=40 + d, **extra)
    g = to_device(inp)
    kw = dict(causal=g["causal"], block_mask=g["block_mask"], kv_len=g["kv_len"],
              scale=g["scale"])
    B, H, N, _ = g["q"].shape
    o, lse = fa.forward(g["q"], g["k"], g["v"], **kw)
    # three upstream gradients whose D = rowsum(dO * O) differ row by row
    dos = [g["do"], (-2.0 * g["do"].float() + 0.25).to(g["do"].dtype),
           torch.flip(g["do"], dims=[2]).contiguous()]
    ws = torch.empty(fa.backward_workspace_bytes(B, H, N, d, g["block_mask"]), device="cuda",
                     dtype=torch.uint8)
    want = one_at_a_time(g, o, lse, dos, ws, kw)
    torch.cuda.synchronize()
    got = [fa.backward(g["q"], g["k"], g["v"], o, lse, do, workspace=ws, **kw)
           for do in dos + dos]
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for i, (dq, dk, dv) in enumerate(got):
        wq, wk, wv = want[i % 3]
        # dK, dV: the same sums in the same order; dQ: fp32 reductions in
        # any order, rounded once
        assert torch.equal(dk, wk) and torch.equal(dv, wv), i
        ref = wq.float().abs().max().item()
        assert (dq.float() - wq.float()).abs().max().item() <= 1e-2 * ref, i
    # the calls' gradients do differ, so a call reading another's D would show
    assert not torch.equal(want[0][1], want[1][1])


def test_back_to_back_packed_calls_see_their_own_preprocess():
    # the packed layout's backward has the same launch chain
    torch.manual_seed(3)
    H, d, lens = 4, 64, [700, 129, 1024]
    total = sum(lens)
    cu = torch.tensor([0, 700, 829, 1853], dtype=torch.int32, device="cuda")
    q, k, v, do = (torch.randn(total, H, d, device="cuda").to(torch.bfloat16) for _ in range(4))
    o, lse = fa.forward_varlen(q, k, v, cu, max(lens), causal=True)
    dos = [do, (0.5 - 3.0 * do.float()).to(torch.bfloat16)]
    ws = torch.empty(fa.varlen_workspace_bytes(len(lens), H, total, max(lens), d), device="cuda",
                     dtype=torch.uint8)
    want = []
    for g in dos:
        torch.cuda.synchronize()
        want.append(tuple(t.clone() for t in fa.backward_varlen(q, k, v, o, lse, g, cu, max(lens),
                                                                causal=True, workspace=ws)))
        torch.cuda.synchronize()
    got = [fa.backward_varlen(q, k, v, o, lse, g, cu, max(lens), causal=True, workspace=ws)
           for g in dos + dos]
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for i, (dq, dk, dv) in enumerate(got):
        wq, wk, wv = want[i % 2]
        assert torch.equal(dk, wk) and torch.equal(dv, wv), i
        ref = wq.float().abs().max().item()
        assert (dq.float() - wq.float()).abs().max().item() <= 1e-2 * ref, i
    assert not torch.equal(want[0][1], want[1][1])


@pytest.mark.parametrize("d,mask", [(64, "causal"), (128, "causal"), (64, "band_global")])
def test_backward_captured_in_a_cuda_graph(d, mask):
    # the backward's kernels carry the programmatic-launch attribute; a
    # stream capture keeps those edges, and replays give the eager results
    extra = dict(global_every=4) if mask == "band_global" else {}
    inp = make_inputs(B=1, H=4, N=1024, d=d, mask=mask, seed=60 + d, **extra)
    g = to_device(inp)
    kw = dict(causal=g["causal"], block_mask=g["block_mask"], scale=g["scale"])
    B, H, N, _ = g["q"].shape
    o, lse = fa.forward(g["q"], g["k"], g["v"], **kw)
    ws = torch.empty(fa.backward_workspace_bytes(B, H, N, d, g["block_mask"]), device="cuda",
                     dtype=torch.uint8)
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
    do = g["do"].clone()
    torch.cuda.synchronize()
    want = [t.clone() for t in fa.backward(g["q"], g["k"], g["v"], o, lse, do, workspace=ws, **kw)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            fa.backward(g["q"], g["k"], g["v"], o, lse, do, workspace=ws, dq=dq, dk=dk, dv=dv,
                        stream=s, **kw)
    torch.cuda.synchronize()
    for scale in (1.0, -0.5):
        do.copy_((g["do"].float() * scale).to(do.dtype))
        graph.replay()
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        ref = [t.clone() for t in fa.backward(g["q"], g["k"], g["v"], o, lse, do, **kw)]
        torch.cuda.synchronize()
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        top = ref[0].float().abs().max().item()
        assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2 * top
        # the replay read the new dO
        assert torch.equal(dk, want[1]) == (scale == 1.0)
