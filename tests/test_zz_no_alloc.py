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
