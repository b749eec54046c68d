"""GPU parity of sliding-window masks (alone and with causal, key padding and
block masks), of scales of either sign and zero, and of the windowed tile
schedule, against the fp64 oracle through the C ABI."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from oracle import attention_forward_rows, live_tiles
from parity import TOL_O, check_close, check_lse, compare_heads, oracle_inputs, run_gpu
from test_gpu_parity import oracle_on_heads

pytestmark = pytest.mark.gpu

WINDOWS = [((0, 0), False), ((5, -1), True), ((100, 0), True), ((128, 128), False),
           ((200, 50), False), ((-1, 64), False), ((300, -1), False), ((127, 1), True)]


@pytest.mark.parametrize("n", [1, 130, 300, 700])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window,causal", WINDOWS)
def test_window_small(n, d, window, causal):
    inp = make_inputs(B=2, H=2, N=n, d=d, mask="none", seed=n + d)
    inp["causal"] = causal
    inp["window"] = window
    heads = [(b, h) for b in range(2) for h in range(2)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)


@pytest.mark.parametrize("d", [64, 128])
def test_window_with_key_padding_and_block_mask(d):
    n = 5 * 128 + 33
    inp = make_inputs(B=3, H=2, N=n, d=d, mask="none", seed=17)
    rng = np.random.default_rng(3)
    bm = (rng.random((6, 6)) < 0.7).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    inp["block_mask"] = bm
    inp["kv_len"] = np.array([n, 200, 0], np.int32)
    inp["causal"] = True
    inp["window"] = (150, -1)
    heads = [(b, h) for b in range(3) for h in range(2)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)


@pytest.mark.parametrize("scale", [-0.09, 0.0, -1e-40])
@pytest.mark.parametrize("d", [64, 128])
def test_scale_of_either_sign_and_zero(scale, d):
    inp = make_inputs(B=1, H=2, N=333, d=d, mask="causal", seed=4)
    inp["scale"] = scale
    inp["window"] = (90, -1)
    heads = [(0, 0), (0, 1)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)


def test_long_sliding_window_sampled_rows():
    # causal sliding window of 1024 keys over 8192 tokens, d = 128
    inp = make_inputs(B=1, H=4, N=8192, d=128, mask="causal", seed=21)
    inp["window"] = (1023, 0)
    res = run_gpu(inp)
    q, k, v, do = oracle_inputs(inp)
    rng = np.random.default_rng(2)
    for h in range(4):
        rows = np.sort(rng.choice(8192, 24, replace=False))
        o, lse = attention_forward_rows(q, k, v, inp["scale"], 0, h, rows, True,
                                        window=(1023, 0))
        check_close("O rows", res["o"][0, h, rows], o, TOL_O)
        check_lse(res["lse"][0, h, rows], lse)
    heads = [(0, 1)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)


@pytest.mark.parametrize("n,causal,window", [(1000, True, (200, 0)), (1000, False, (0, 0)),
                                             (777, False, (128, 300)), (4096, True, (1023, -1)),
                                             (300, False, (-1, 5))])
def test_tile_schedule_with_window(n, causal, window):
    t = (n + 127) // 128
    rp, ci, pf = fa.tile_schedule(n, causal, window=window)
    rp, ci, pf = rp.cpu().numpy(), ci.cpu().numpy(), pf.cpu().numpy()
    want = live_tiles(n, causal, window=window)
    got = {}
    for qt in range(t):
        for e in range(rp[qt], rp[qt + 1]):
            got[(qt, int(ci[e]))] = int(pf[e])
    assert got == want
