"""The persistent dK/dV kernel at d = 64 (padded layout, no dropout): one CTA
per SM walking work items taken from a counter in the workspace.  What the
schedule adds over one CTA per key tile is checked here: several items per
CTA (the K/V buffers, item buffers and step barriers carried from one item
to the next), items with no step at all (key tiles past a batch element's
key length), split parts of heavy key tiles, the counter's reset by each
call's preprocess, and that the dynamic assignment of items to CTAs leaves
dK and dV bit-for-bit the same from call to call.  Marked ``gpu``."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from parity import compare_heads, run_gpu, to_device
from test_gpu_parity import oracle_on_heads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_many_items_per_cta(causal):
    # 4 x 16 heads x 12 key tiles = 768 items, about five per SM; N not a
    # multiple of 128, so every head's last item has one 64-row step
    inp = make_inputs(B=4, H=16, N=1472, d=64, mask="causal" if causal else "none", seed=90)
    res = run_gpu(inp)
    heads = [(0, 0), (1, 7), (2, 15), (3, 3)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)


def test_items_without_steps():
    # key lengths of 0 and of less than a tile: most key tiles of those
    # batch elements have no step; their dK, dV rows must come out 0
    inp = make_inputs(B=8, H=4, N=1024, d=64, mask="none", seed=91)
    inp["kv_len"] = np.array([1024, 0, 77, 1024, 0, 513, 128, 1], np.int32)
    res = run_gpu(inp)
    heads = [(b, h) for b in range(8) for h in (0, 3)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)
    assert np.all(res["dk"][1] == 0) and np.all(res["dv"][1] == 0)
    assert np.all(res["dk"][2][:, 128:] == 0) and np.all(res["dv"][2][:, 128:] == 0)


def test_split_items_across_ctas():
    # a band + global-column mask with the split workspace: the global
    # columns run as parts on different CTAs, the join adds them
    inp = make_inputs(B=2, H=16, N=4096, d=64, mask="band_global", seed=92, global_every=8)
    g = to_device(inp)
    B, H, N, d = g["q"].shape
    assert fa.backward_workspace_bytes(B, H, N, d, g["block_mask"]) > \
        fa.backward_workspace_bytes(B, H, N, d)
    res = run_gpu(inp)
    heads = [(0, 0), (1, 9)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)


def test_counter_reset_and_repeatability():
    # three calls on one workspace: each call's preprocess clears the
    # counter (a stale counter would leave items unrun), and dK, dV repeat
    # bit for bit however the items fell to the CTAs
    inp = make_inputs(B=4, H=12, N=1024, d=64, mask="causal", seed=93)
    g = to_device(inp)
    B, H, N, d = g["q"].shape
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=True)
    ws = torch.empty(fa.backward_workspace_bytes(B, H, N, d), device="cuda", dtype=torch.uint8)
    outs = []
    for _ in range(3):
        dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True,
                                 workspace=ws)
        outs.append((dq.clone(), dk.clone(), dv.clone()))
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for dq, dk, dv in outs[1:]:
        assert torch.equal(dk, outs[0][1]) and torch.equal(dv, outs[0][2])
        ref = outs[0][0].float().abs().max().item()
        assert (dq.float() - outs[0][0].float()).abs().max().item() <= 1e-2 * ref
    heads = [(0, 0), (3, 11)]
    res = {"o": o.double().cpu().numpy(), "lse": lse.double().cpu().numpy(),
           "dq": outs[2][0].double().cpu().numpy(), "dk": outs[2][1].double().cpu().numpy(),
           "dv": outs[2][2].double().cpu().numpy()}
    compare_heads(res, oracle_on_heads(inp, heads), heads)
