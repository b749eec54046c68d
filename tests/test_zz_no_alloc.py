"""The allocation-free backward (``fa_backward_noalloc``): for callers that
cannot allocate device memory and so cannot pass a workspace, the library
runs the same backward in a fixed scratch array of its own.  Checked here
against the workspace entry point (``fa_backward``) on the same inputs, on
two calls in a row (the scratch keeps the previous call's contents, so the
second call shows that nothing stale is read).  Collected last on purpose."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from parity import TOL_GRAD, check_close, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,mask", [(64, "causal"), (128, "none")])
def test_noalloc_backward_matches_workspace_backward(d, mask):
    for call, seed in enumerate((21, 22)):
        inp = make_inputs(B=2, H=3, N=700 + 100 * call, d=d, mask=mask, seed=seed)
        g = to_device(inp)
        kw = dict(causal=g["causal"], scale=g["scale"])
        o, lse = fa.forward(g["q"], g["k"], g["v"], **kw)
        want = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], **kw)
        got = fa.backward_noalloc(g["q"], g["k"], g["v"], o, lse, g["do"], **kw)
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        for name, a, b in zip(("dQ", "dK", "dV"), got, want):
            check_close(f"{name} (call {call})", a.double().cpu().numpy(),
                        b.double().cpu().numpy(), TOL_GRAD)


def test_noalloc_rejects_problems_beyond_its_scratch():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    need = fa.backward_workspace_bytes(64, 16, 8192, 128)
    assert need > fa.NOALLOC_SCRATCH_BYTES
    lib = fa.load()
    p = fa._ptr(q)
    st = lib.fa_backward_noalloc(p, p, p, p, fa._ptr(lse), p, p, p, p, 64, 16, 8192, 128,
                                 0.1, 0, None, None, fa._stream())
    assert st == fa.FA_ERR_INVALID_ARG


def test_noalloc_block_mask_against_the_oracle():
    # A block mask with global key columns: the array's room beyond the base
    # workspace lets the backward split those heavy key tiles (plan items and
    # fp32 part slots in the shared array).  Two calls in a row with
    # different masks and inputs, each against the fp64 oracle and against
    # fa_backward given the masked (split) workspace.
    from exact_io_aware_tma_gb300.workloads import band_global_block_mask, to_f64
    from oracle import attention_backward
    B, H, N, d = 1, 2, 1024, 64
    T = N // 128
    for call, (seed, band, every) in enumerate(((23, 1, 4), (24, 0, 3))):
        bm_np = band_global_block_mask(T, band, every)
        inp = make_inputs(B=B, H=H, N=N, d=d, mask="none", seed=seed)
        g = to_device(inp)
        bm = torch.from_numpy(bm_np).cuda()
        assert fa.backward_workspace_bytes(B, H, N, d, bm) <= fa.NOALLOC_SCRATCH_BYTES
        o, lse = fa.forward(g["q"], g["k"], g["v"], block_mask=bm, scale=g["scale"])
        got = fa.backward_noalloc(g["q"], g["k"], g["v"], o, lse, g["do"], block_mask=bm,
                                  scale=g["scale"])
        ws = torch.empty(fa.backward_workspace_bytes(B, H, N, d, bm), device="cuda",
                         dtype=torch.uint8)
        want = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], block_mask=bm,
                           scale=g["scale"], workspace=ws)
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        q, k, v, do = (to_f64(inp[x]) for x in ("q", "k", "v", "do"))
        ref = attention_backward(q, k, v, do, inp["scale"], False, bm_np, None)
        for name, a, b, r in zip(("dQ", "dK", "dV"), got, want, ref[:3]):
            a = a.double().cpu().numpy()
            check_close(f"{name} vs oracle (call {call})", a, r, TOL_GRAD)
            check_close(f"{name} vs fa_backward (call {call})", a, b.double().cpu().numpy(),
                        TOL_GRAD)
