"""Failure detection without a GPU fault: the bounded mbarrier waits.

Every wait in the attention kernels gives up after a time limit, records
FA_ERR_TIMEOUT in the library's device error word, stops the rest of its
CTA, lets the CTA's copies and tensor-core work in flight finish and frees
its tensor memory.  The self-test entry points run the d = 128 forward and
dK/dV kernels, and the persistent d = 64 dK/dV kernel, with one arrival
withheld on purpose (one warp per CTA skips one signal) and a 1 ms limit,
so that path runs: the status must come back as FA_ERR_TIMEOUT within a
fraction of a second, be cleared by reading it, and a normal forward +
backward on the same stream afterwards must return FA_OK and match the
fp64 oracle.  Nothing here faults, traps or hangs the
GPU: every wait involved is bounded and every copy issued completes."""

import time

import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from oracle import attention_backward
from parity import (TOL_GRAD, TOL_O, check_close, check_lse, oracle_inputs, to_device)

pytestmark = pytest.mark.gpu


def run_lost_signal(which, g, B, H, N, d):
    lib = fa.load()
    P = fa._ptr
    o = torch.empty_like(g["q"])
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    sp = fa._stream()
    if which == "forward":
        st = lib.fa_selftest_forward_lost_signal(P(g["q"]), P(g["k"]), P(g["v"]), P(o), P(lse),
                                                 B, H, N, d, g["scale"], int(g["causal"]), sp)
    else:
        # a correct forward first (its O and LSE feed the backward)
        o, lse = fa.forward(g["q"], g["k"], g["v"], causal=g["causal"], scale=g["scale"])
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        wsb = fa.backward_workspace_bytes(B, H, N, d)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        st = lib.fa_selftest_backward_lost_signal(
            P(g["q"]), P(g["k"]), P(g["v"]), P(o), P(lse), P(g["do"]), P(dq), P(dk), P(dv),
            B, H, N, d, g["scale"], int(g["causal"]), P(ws), wsb, sp)
    return st


@pytest.mark.parametrize("which,d", [("forward", 128), ("forward", 64), ("backward", 128),
                                     ("backward", 64)])
def test_withheld_arrival_times_out_and_the_device_stays_usable(which, d):
    # backward d = 64: more work items (B*H*T = 192) than persistent CTAs
    # (one per SM), so the CTAs abort with items still to fetch; forward
    # d = 64: two one-tile CTAs per SM, each aborting with the next S issued
    # and its stage loads in flight
    B, H, N = (1, 4, 1024) if d == 128 else (2, 12, 1024)
    inp = make_inputs(B=B, H=H, N=N, d=d, mask="causal", seed=41)
    g = to_device(inp)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK  # nothing pending from earlier tests

    t0 = time.perf_counter()
    st = run_lost_signal(which, g, B, H, N, d)
    assert st == fa.FA_OK, fa.status_string(st)
    status = fa.last_device_status()
    elapsed = time.perf_counter() - t0
    assert status == fa.FA_ERR_TIMEOUT, fa.status_string(status)
    # one wave of CTAs, each giving up after 1 ms (not the 2 s product limit)
    assert elapsed < 1.0, elapsed
    # reading the status cleared it
    assert fa.last_device_status() == fa.FA_OK

    # the same stream, a normal call: FA_OK and the oracle's results
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=True, scale=g["scale"])
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True,
                             scale=g["scale"])
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    q, k, v, do = oracle_inputs(inp)
    rdq, rdk, rdv, ro, rlse, _ = attention_backward(q, k, v, do, inp["scale"], causal=True)
    check_close("O", o.double().cpu().numpy(), ro, TOL_O)
    check_lse(lse.double().cpu().numpy(), rlse)
    for name, got, want in (("dQ", dq, rdq), ("dK", dk, rdk), ("dV", dv, rdv)):
        check_close(name, got.double().cpu().numpy(), want, TOL_GRAD)


def test_lost_signal_entry_points_reject_other_head_dims():
    lib = fa.load()
    x = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    P = fa._ptr
    st = lib.fa_selftest_forward_lost_signal(P(x), P(x), P(x), P(x), P(lse), 1, 1, 128, 96,
                                             0.125, 1, fa._stream())
    assert st == fa.FA_ERR_UNSUPPORTED
