"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the fp64 oracle at the tolerances of the method's
statement of correctness (exact up to floating-point reordering; bf16
inputs, fp32 accumulation):

  O           : max |gpu - ref| <= 1e-2 * max |ref|
  dQ, dK, dV  : max |gpu - ref| <= 2e-2 * max |ref|
  LSE         : max |gpu - ref| <= 1e-3 on rows with an allowed key;
                exactly -inf (and O == 0) on rows without one.

When a reference tensor is identically zero (dQ and dK when every row has a
single allowed key, where dS = P (dP - D) vanishes), the relative bound has
nothing to scale; the bound then uses max |ref| floored at ABS_FLOOR.  The
floor comes from the arithmetic of that cancellation: dP_ij and D_i are two
fp32 dot products of d bf16 products of N(0, 1) values (magnitude
sum_c |dO_c V_c| ~ 0.64 d ~ 80 at d = 128), each off by about sqrt(d) * 2^-24
times that (~5e-5), so dS ~ 5e-5 and dQ = scale * dS K ~ 0.09 * 5e-5 * 3
~ 1e-5.  ABS_FLOOR = 1e-3 puts the bound (2e-5 for gradients) above that
noise and still two orders of magnitude below every nonzero gradient
magnitude in the tests (max |dQ| is O(0.1) or more).
"""

import numpy as np
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import to_f64

TOL_O, TOL_GRAD, TOL_LSE = 1e-2, 2e-2, 1e-3
ABS_FLOOR = 1e-3


def to_device(inp, dev="cuda"):
    out = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if inp["block_mask"] is not None:
        out["block_mask"] = torch.from_numpy(inp["block_mask"]).to(dev)
    if inp["kv_len"] is not None:
        out["kv_len"] = torch.from_numpy(inp["kv_len"]).to(dev)
    return out


def run_gpu(inp, backward=True):
    g = to_device(inp)
    drop = inp.get("dropout")
    kw = dict(causal=g["causal"], block_mask=g["block_mask"], kv_len=g["kv_len"],
              scale=g["scale"], window=inp.get("window"),
              dropout=None if drop is None else (drop["p"], drop["seed"], drop["offset"]))
    o, lse = fa.forward(g["q"], g["k"], g["v"], **kw)
    res = dict(o=o, lse=lse)
    if backward:
        dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], **kw)
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    return {k: v.double().cpu().numpy() for k, v in res.items()}


def oracle_inputs(inp):
    return (to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]),
            None if inp["do"] is None else to_f64(inp["do"]))


def check_close(name, got, want, tol):
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    ref = max(np.abs(want).max(), ABS_FLOOR)
    err = np.abs(got - want).max()
    assert err <= tol * ref, f"{name}: max err {err:.3e} > {tol} * {ref:.3e}"
    return err / ref


def check_lse(got, want):
    live = np.isfinite(want)
    assert np.array_equal(np.isneginf(got), ~live), "LSE: -inf rows differ"
    if live.any():
        err = np.abs(got[live] - want[live]).max()
        assert err <= TOL_LSE, f"LSE: max abs err {err:.3e}"
        return err
    return 0.0


def compare_heads(res, ref, heads, backward=True):
    """Compare GPU results with oracle results on the listed (b, h) heads."""
    rdq, rdk, rdv, ro, rlse = ref
    out = {}
    sel = tuple(np.array(x) for x in zip(*heads))
    out["o"] = check_close("O", res["o"][sel], ro[sel], TOL_O)
    out["lse"] = check_lse(res["lse"][sel], rlse[sel])
    dead = np.isneginf(rlse[sel])
    assert np.all(res["o"][sel][dead] == 0.0), "O must be 0 on rows without an allowed key"
    if backward:
        out["dq"] = check_close("dQ", res["dq"][sel], rdq[sel], TOL_GRAD)
        out["dk"] = check_close("dK", res["dk"][sel], rdk[sel], TOL_GRAD)
        out["dv"] = check_close("dV", res["dv"][sel], rdv[sel], TOL_GRAD)
    return out
