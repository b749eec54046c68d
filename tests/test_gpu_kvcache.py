"""GPU parity of attention against a key/value cache (split kernel + merge)
and of the standalone merge, through the C ABI, against the fp64 oracle.
Tolerances as for the forward pass: O within 1e-2 * max|ref|, LSE within
1e-3 absolute, rows without an allowed key exactly O = 0, LSE = -inf."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import (KVCACHE_WORKLOADS, kvcache_workload_inputs,
                                                make_kvcache_inputs, to_f64)
from oracle import attention_forward_kvcache, merge_partial_states
from parity import TOL_O, check_close, check_lse

pytestmark = pytest.mark.gpu


def run_kvcache(inp, num_splits=0, k=None, v=None):
    dev = "cuda"
    q = inp["q"].to(dev)
    kk = (inp["k"] if k is None else k).to(dev)
    vv = (inp["v"] if v is None else v).to(dev)
    cl = None if inp["cache_len"] is None else torch.from_numpy(inp["cache_len"]).to(dev)
    o, lse = fa.forward_kvcache(q, kk, vv, cache_len=cl, causal=inp["causal"],
                                scale=inp["scale"], num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_heads(inp, heads=None):
    q, k, v = to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"])
    B, H = q.shape[:2]
    if heads is None:
        return attention_forward_kvcache(q, k, v, inp["scale"], inp["causal"], inp["cache_len"])
    o = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:3], np.nan)
    for b, h in heads:
        cl = None if inp["cache_len"] is None else inp["cache_len"][b:b + 1]
        r = attention_forward_kvcache(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                      v[b:b + 1, h:h + 1], inp["scale"], inp["causal"], cl)
        o[b, h], lse[b, h] = r[0][0, 0], r[1][0, 0]
    return o, lse


def compare(got, want, heads=None):
    (go, gl), (wo, wl) = got, want
    if heads is not None:
        sel = tuple(np.array(x) for x in zip(*heads))
        go, gl, wo, wl = go[sel], gl[sel], wo[sel], wl[sel]
    check_close("O", go, wo, TOL_O)
    check_lse(gl, wl)
    assert np.all(go[np.isneginf(wl)] == 0.0)


CASES = [
    # B, H, Nq, Nk, d, causal, cache lengths (None = all slots), splits
    (2, 3, 1, 1, 64, False, None, 1),
    (2, 3, 1, 63, 128, False, [63, 1], 1),
    (2, 3, 1, 65, 64, False, [65, 64], 3),
    (2, 3, 2, 200, 128, True, [200, 2], 0),
    (3, 2, 3, 1000, 64, True, [1000, 0, 513], 0),
    (3, 2, 4, 1000, 128, True, [999, 3, 64], 7),
    (2, 2, 5, 777, 64, True, [777, 4], 0),
    (2, 2, 8, 4096, 128, False, [4096, 2000], 0),
    (2, 2, 1, 3000, 64, False, [5000, -3], 64),    # lengths clamped to [0, Nk]
    (1, 4, 2, 130, 128, False, [130], 256),        # more splits than key tiles
    (2, 1, 6, 300, 64, False, None, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_small_cases(case):
    B, H, Nq, Nk, d, causal, lens, S = case
    inp = make_kvcache_inputs(B, H, Nq, Nk, d, causal=causal, seed=B * 100 + Nk)
    if lens is not None:
        inp["cache_len"] = np.array(lens, np.int32)
    compare(run_kvcache(inp, S), oracle_heads(inp))


@pytest.mark.parametrize("d", [64, 128])
def test_slots_past_the_cache_length_are_never_used(d):
    # Non-finite garbage in K and V past cache_len must not reach the result.
    inp = make_kvcache_inputs(2, 2, 3, 500, d, causal=True, seed=3)
    inp["cache_len"] = np.array([300, 131], np.int32)
    k, v = inp["k"].clone(), inp["v"].clone()
    for b, L in enumerate(inp["cache_len"]):
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("inf")
    compare(run_kvcache(inp, 0, k, v), oracle_heads(inp))


def test_split_count_does_not_change_the_result_beyond_rounding():
    inp = make_kvcache_inputs(2, 4, 1, 5000, 128, seed=8)
    want = oracle_heads(inp)
    for S in (1, 2, 5, 19, 78):
        compare(run_kvcache(inp, S), want)


@pytest.mark.parametrize("name", list(KVCACHE_WORKLOADS))
def test_workloads_sampled_heads(name):
    inp = kvcache_workload_inputs(name)
    B, H = inp["q"].shape[:2]
    rng = np.random.default_rng(1)
    heads = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, B, 6), rng.integers(0, H, 6))}
                   | {(0, 0), (B - 1, H - 1)})
    compare(run_kvcache(inp, 0), oracle_heads(inp, heads), heads)


@pytest.mark.parametrize("S,rows,d", [(1, 10, 64), (3, 100, 128), (17, 33, 4), (5, 7, 1024),
                                      (2, 1000, 96)])
def test_combine_matches_oracle_merge(S, rows, d):
    rng = np.random.default_rng(S * rows + d)
    op = rng.standard_normal((S, rows, d)).astype(np.float32)
    lp = (6.0 * rng.standard_normal((S, rows))).astype(np.float32)
    lp[rng.random((S, rows)) < 0.2] = -np.inf
    lp[:, 0] = -np.inf                       # a row whose parts are all empty
    o, lse = fa.combine(torch.from_numpy(op).cuda(), torch.from_numpy(lp).cuda())
    torch.cuda.synchronize()
    wo, wl = merge_partial_states(op.astype(np.float64), lp.astype(np.float64))
    check_close("O", o.double().cpu().numpy(), wo, TOL_O)
    check_lse(lse.double().cpu().numpy(), wl)
    assert torch.all(o[0] == 0)


def test_repeat_calls_are_identical():
    inp = make_kvcache_inputs(4, 4, 2, 3000, 64, causal=True, seed=2)
    a = run_kvcache(inp, 0)
    b = run_kvcache(inp, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
