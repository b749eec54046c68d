"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded inputs.  Marked ``gpu``."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import (WORKLOADS, make_inputs,
                                                workload_inputs, to_f64)
from oracle import attention_backward, attention_forward_rows, dropout_p8, live_tiles
from parity import (TOL_GRAD, TOL_O, check_close, check_lse, compare_heads,
                    oracle_inputs, run_gpu, to_device)

pytestmark = pytest.mark.gpu


def oracle_on_heads(inp, heads):
    """Oracle fwd+bwd of the listed (b, h) heads, returned at full shape."""
    q, k, v, do = oracle_inputs(inp)
    B, H, N, d = q.shape
    out = [np.full(q.shape, np.nan) for _ in range(4)] + [np.full((B, H, N), np.nan)]
    for b, h in heads:
        kv = None if inp["kv_len"] is None else inp["kv_len"][b:b + 1]
        sl = (slice(b, b + 1), slice(h, h + 1))
        drop = inp.get("dropout")
        drop = None if drop is None else dict(p8=dropout_p8(drop["p"]), seed=drop["seed"],
                                              offset=drop["offset"], bh0=b * H + h)
        r = attention_backward(q[sl], k[sl], v[sl], do[sl], inp["scale"], inp["causal"],
                               inp["block_mask"], kv, window=inp.get("window"), dropout=drop)
        for arr, val in zip(out, (r[0], r[1], r[2], r[3], r[4])):
            arr[b, h] = val[0, 0]
    return tuple(out)


# Full-size workloads.  Heads the oracle recomputes in full: every head of the
# small workloads, a few of the large ones (the rest are covered by sampled
# rows and gradient invariants below).
HEADS = {
    "tiny_dense_n128_d64": "all",
    "bert_large_keypad_n512_d64": "all",
    "gpt2_causal_n1024_d64": "all",
    "long_causal_n8192_d128": [(0, 0), (1, 15), (1, 6)],
    "block_sparse_n16384_d64": [(0, 0), (0, 5)],
}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_parity(name):
    inp = workload_inputs(name)
    B, H = inp["q"].shape[:2]
    heads = HEADS[name]
    heads = [(b, h) for b in range(B) for h in range(H)] if heads == "all" else heads
    res = run_gpu(inp)
    ref = oracle_on_heads(inp, heads)
    compare_heads(res, ref, heads)


@pytest.mark.parametrize("name", ["long_causal_n8192_d128", "block_sparse_n16384_d64"])
def test_workload_sampled_rows_and_invariants(name):
    # Every head: 16 sampled query rows of O / LSE against the oracle, and
    # the exact gradient identities sum_j dK_j = 0, sum_j dV_j = sum_i dO_i.
    inp = workload_inputs(name)
    res = run_gpu(inp)
    q, k, v, do = oracle_inputs(inp)
    B, H, N, d = q.shape
    rng = np.random.default_rng(0)
    for b in range(B):
        for h in range(H):
            rows = np.sort(rng.choice(N, 16, replace=False))
            rows[0], rows[-1] = 0, N - 1
            o, lse = attention_forward_rows(q, k, v, inp["scale"], b, h, rows,
                                            inp["causal"], inp["block_mask"], inp["kv_len"])
            check_close("O rows", res["o"][b, h, rows], o, TOL_O)
            check_lse(res["lse"][b, h, rows], lse)
    dk_sum = res["dk"].sum(axis=2)
    dv_sum = res["dv"].sum(axis=2)
    do_sum = do.sum(axis=2)
    # bf16 rounding of each dK / dV element bounds the sums' drift
    scale_k = np.abs(res["dk"]).max() * np.sqrt(N)
    assert np.abs(dk_sum).max() <= 1e-2 * scale_k
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * np.abs(do_sum).max() + 1e-2 * np.sqrt(N)


SMALL = [(n, d) for n in (1, 7, 128, 130, 255) for d in (64, 128)]
MASKS = ["none", "causal", "kv_len", "block", "causal_kv", "block_causal_kv"]


def small_inputs(n, d, mask, B=2, H=3, seed=11):
    kind = {"none": "none", "causal": "causal"}.get(mask, "none")
    inp = make_inputs(B=B, H=H, N=n, d=d, mask=kind, seed=seed)
    rng = np.random.default_rng(seed + n + d)
    if "causal" in mask:
        inp["causal"] = True
    if "kv" in mask:
        inp["kv_len"] = rng.integers(0, n + 2, size=B).astype(np.int32)
        inp["kv_len"][0] = max(1, n // 2)
    if "block" in mask:
        t = (n + 127) // 128
        bm = (rng.random((t, t)) < 0.6).astype(np.uint8)
        np.fill_diagonal(bm, 1)
        inp["block_mask"] = bm
    return inp


@pytest.mark.parametrize("n,d", SMALL)
@pytest.mark.parametrize("mask", MASKS)
def test_small_shapes(n, d, mask):
    inp = small_inputs(n, d, mask)
    res = run_gpu(inp)
    heads = [(b, h) for b in range(2) for h in range(3)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)


@pytest.mark.parametrize("d", [64, 128])
def test_multi_tile_block_mask_with_dead_rows(d):
    # 5 query tiles with a ragged tail; query tile 2 has no live key tile, so
    # its rows must give O = 0, LSE = -inf and no gradient; kv_len = 0 kills
    # a whole batch element.
    n = 4 * 128 + 77
    inp = make_inputs(B=3, H=2, N=n, d=d, mask="none", seed=5)
    bm = np.ones((5, 5), np.uint8)
    bm[2, :] = 0
    bm[0, 3] = 0
    bm[4, 1] = 0
    inp["block_mask"] = bm
    inp["kv_len"] = np.array([n, 0, 300], np.int32)
    res = run_gpu(inp)
    heads = [(b, h) for b in range(3) for h in range(2)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)
    assert np.all(res["o"][:, :, 256:384] == 0) and np.all(np.isneginf(res["lse"][:, :, 256:384]))
    assert np.all(res["o"][1] == 0) and np.all(res["dk"][1] == 0) and np.all(res["dq"][1] == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_larger_scores_stay_exact(d):
    # Scaled-up inputs push the running max through many rescalings.
    inp = make_inputs(B=1, H=2, N=700, d=d, mask="causal", seed=9)
    for x in ("q", "k"):
        inp[x] = (inp[x].float() * 3.0).to(torch.bfloat16)
    res = run_gpu(inp)
    heads = [(0, 0), (0, 1)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)


def test_forward_is_deterministic_and_stream_aware():
    inp = make_inputs(B=2, H=4, N=1000, d=64, mask="causal", seed=3)
    g = to_device(inp)
    o1, l1 = fa.forward(g["q"], g["k"], g["v"], causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = fa.forward(g["q"], g["k"], g["v"], causal=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("n,causal,kind", [
    (1000, True, None), (1000, False, "kv"), (16384, False, "band"),
    (8192, True, None), (333, True, "kv"), (1, False, None), (900, True, "block")])
def test_tile_schedule_bit_exact(n, causal, kind):
    from exact_io_aware_tma_gb300.workloads import band_global_block_mask
    t = (n + 127) // 128
    bm = kv = None
    if kind == "band":
        bm = band_global_block_mask(t)
    if kind == "block":
        bm = (np.random.default_rng(n).random((t, t)) < 0.5).astype(np.uint8)
    if kind == "kv":
        kv = np.array([n, 5, n // 3, 0], np.int32)
    for b in range(1 if kv is None else len(kv)):
        rp, ci, pf = fa.tile_schedule(
            n, causal, None if bm is None else torch.from_numpy(bm).cuda(),
            None if kv is None else torch.from_numpy(kv).cuda(), b)
        rp, ci, pf = rp.cpu().numpy(), ci.cpu().numpy(), pf.cpu().numpy()
        want = live_tiles(n, causal, bm, None if kv is None else int(kv[b]))
        got = {}
        for qt in range(t):
            for e in range(rp[qt], rp[qt + 1]):
                got[(qt, int(ci[e]))] = int(pf[e])
        assert got == want
        assert rp[t] == len(want)
        # query-tile-major, ascending key tiles inside a row
        assert all(np.all(np.diff(ci[rp[qt]:rp[qt + 1]]) > 0) for qt in range(t))


def test_invalid_arguments_on_device():
    q = torch.zeros(1, 1, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward(q, q, q)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    assert fa.last_device_status() == fa.FA_OK


@pytest.mark.parametrize("n,causal,kv", [(300, False, True), (300, True, False), (640, True, True),
                                         (384, False, False)])
def test_d64_grids_over_one_wave(n, causal, kv):
    # d = 64 with one to four query-tile pairs per SM: odd tile counts (a
    # pair with one tile), key lengths of 0 (pairs with no live key tile,
    # whose O must be 0 even though its TMEM columns were never written) and
    # short ones
    T = (n + 127) // 128
    B, H = 4, (200 + 4 * ((T + 1) // 2) - 1) // (4 * ((T + 1) // 2))
    assert 152 < B * H * ((T + 1) // 2) <= 4 * 152
    inp = make_inputs(B=B, H=H, N=n, d=64, mask="causal" if causal else "none", seed=n + H)
    if kv:
        inp["kv_len"] = np.array([n, 0, n // 3, 129], np.int32)
    res = run_gpu(inp)
    heads = [(b, h) for b in range(B) for h in range(0, H, 7)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)
    if kv:
        assert np.all(res["o"][1] == 0) and np.all(np.isneginf(res["lse"][1]))
