"""GPU parity of dropout on P (mask regenerated from Philox4x32-10 in both
passes) against the fp64 oracle through the C ABI: the keep mask itself bit
for bit, read off the forward (V = identity) and the backward (dO =
identity), and O / LSE / gradients within the usual tolerances."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs, to_f64
from oracle import attention_backward_varlen, dropout_keep, dropout_p8
from parity import TOL_GRAD, TOL_O, check_close, check_lse, compare_heads, run_gpu
from test_gpu_parity import oracle_on_heads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("p_drop,seed,offset", [(0.1, 7, 0), (0.5, 2**40 + 3, 17), (0.9, 5, 2)])
def test_forward_mask_bit_exact(d, p_drop, seed, offset):
    # N = d and V = I: O[i, c] = P[i, c] Z[i, c] / (1 - p), so O == 0 exactly
    # where the element was dropped (P > 0 everywhere without a mask).
    B, H, N = 2, 3, d
    inp = make_inputs(B=B, H=H, N=N, d=d, mask="none", seed=d)
    q, k = (inp[x].cuda() for x in ("q", "k"))
    v = torch.eye(N, dtype=torch.bfloat16, device="cuda").expand(B, H, N, d).contiguous()
    o, _ = fa.forward(q, k, v, dropout=(p_drop, seed, offset))
    torch.cuda.synchronize()
    o = o.float().cpu().numpy()
    p8 = dropout_p8(p_drop)
    for b in range(B):
        for h in range(H):
            keep = dropout_keep(seed, offset, p8, b * H + h, np.arange(N), np.arange(N))
            assert np.array_equal(o[b, h] != 0, keep), (b, h)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_mask_bit_exact(d):
    # dO = I (N = d): dV[j, c] = P[c, j] Z[c, j] / (1 - p): the backward's
    # regenerated mask, transposed, is the zero pattern of dV.
    B, H, N = 2, 2, d
    p_drop, seed, offset = 0.3, 123456789, 9
    inp = make_inputs(B=B, H=H, N=N, d=d, mask="none", seed=d + 1)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    do = torch.eye(N, dtype=torch.bfloat16, device="cuda").expand(B, H, N, d).contiguous()
    o, lse = fa.forward(q, k, v, dropout=(p_drop, seed, offset))
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, dropout=(p_drop, seed, offset))
    torch.cuda.synchronize()
    dv = dv.float().cpu().numpy()
    p8 = dropout_p8(p_drop)
    for b in range(B):
        for h in range(H):
            keep = dropout_keep(seed, offset, p8, b * H + h, np.arange(N), np.arange(N))
            assert np.array_equal(dv[b, h] != 0, keep.T), (b, h)


SHAPES = [(1, 64), (130, 64), (300, 128), (513, 128)]


@pytest.mark.parametrize("n,d", SHAPES)
@pytest.mark.parametrize("causal,window", [(False, None), (True, None), (True, (100, 0))])
@pytest.mark.parametrize("p_drop", [0.1, 0.5])
def test_dropout_parity(n, d, causal, window, p_drop):
    inp = make_inputs(B=2, H=2, N=n, d=d, mask="none", seed=n * 3 + d)
    inp["causal"] = causal
    inp["window"] = window
    inp["dropout"] = dict(p=p_drop, seed=1000 + n, offset=3)
    heads = [(b, h) for b in range(2) for h in range(2)]
    res, ref = run_gpu(inp), oracle_on_heads(inp, heads)
    if n > 1:
        compare_heads(res, ref, heads)
        return
    # One key per row: dS = P (z dP - D) cancels exactly, so the exact dQ and
    # dK are 0, while the GPU's D comes from the bf16 O = z V (no longer
    # exact once scaled by z = 1/(1-p)): |D error| <= 2^-8 sum_c |dO_c O_c|,
    # hence |dQ|, |dK| <= scale * 2^-8 * max sum_c |dO_c O_c| * max |K, Q|.
    # O, LSE and dV keep the usual relative bounds.
    compare_heads({k_: v_ for k_, v_ in res.items()}, ref, heads, backward=False)
    check_close("dV", res["dv"], ref[2], TOL_GRAD)
    do, o = to_f64(inp["do"]), ref[3]
    bound = abs(inp["scale"]) * 2.0 ** -8 * np.abs(do * o).sum(-1).max() * max(
        np.abs(to_f64(inp["k"])).max(), np.abs(to_f64(inp["q"])).max())
    assert np.abs(res["dq"]).max() <= bound and np.abs(res["dk"]).max() <= bound


def test_dropout_long_causal_head():
    inp = make_inputs(B=1, H=2, N=2048, d=128, mask="causal", seed=31)
    inp["dropout"] = dict(p=0.1, seed=99, offset=1)
    heads = [(0, 0), (0, 1)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)


def test_dropout_packed_sequences():
    lens = [300, 1, 200, 513]
    H, d = 2, 64
    g = torch.Generator(device="cpu").manual_seed(4)
    total = sum(lens)
    q, k, v, do = (torch.randn((total, H, d), generator=g).to(torch.bfloat16) for _ in range(4))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    drop = (0.2, 77, 5)
    gq, gk, gv, gdo = (t.cuda() for t in (q, k, v, do))
    gcu = torch.from_numpy(cu).cuda()
    o, lse = fa.forward_varlen(gq, gk, gv, gcu, max(lens), causal=True, dropout=drop)
    dq, dk, dv = fa.backward_varlen(gq, gk, gv, o, lse, gdo, gcu, max(lens), causal=True,
                                    dropout=drop)
    torch.cuda.synchronize()
    ref = attention_backward_varlen(to_f64(q), to_f64(k), to_f64(v), to_f64(do), cu,
                                    1 / np.sqrt(d), True, None,
                                    dict(p8=dropout_p8(0.2), seed=77, offset=5))
    got = [t.double().cpu().numpy() for t in (dq, dk, dv, o, lse)]
    for name, g_, r_, tol in (("dQ", got[0], ref[0], TOL_GRAD), ("dK", got[1], ref[1], TOL_GRAD),
                              ("dV", got[2], ref[2], TOL_GRAD), ("O", got[3], ref[3], TOL_O)):
        check_close(name, g_, r_, tol)
    check_lse(got[4], ref[4])


def test_dropout_is_reproducible_and_seeded():
    inp = make_inputs(B=1, H=2, N=256, d=64, mask="causal", seed=8)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    a, _ = fa.forward(q, k, v, causal=True, dropout=(0.3, 5, 0))
    b, _ = fa.forward(q, k, v, causal=True, dropout=(0.3, 5, 0))
    c, _ = fa.forward(q, k, v, causal=True, dropout=(0.3, 5, 1))
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


def test_dropout_probability_is_validated():
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    for p in (1.0, -0.1, float("nan")):
        with pytest.raises(fa.FAError) as e:
            fa.forward(q, q, q, dropout=(p, 0, 0))
        assert e.value.status == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("n", [2048, 2176])
def test_dropout_d64_on_both_sides_of_the_cta_shape_threshold(n):
    # at d = 64 with dropout the forward runs one query tile per CTA up to
    # 2048 rows and a pair of query tiles per CTA beyond: both match
    inp = make_inputs(B=1, H=1, N=n, d=64, mask="causal", seed=n)
    inp["dropout"] = dict(p=0.15, seed=4242, offset=7)
    heads = [(0, 0)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)
