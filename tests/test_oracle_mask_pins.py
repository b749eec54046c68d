"""Pins for the oracle's sliding-window masks and packed variable-length
sequences.  CPU only.

Checks: (a) closed forms of narrow windows, (b) brute force with scalar loops,
(c) torch SDPA / autograd in fp64 with an explicit boolean mask (for packed
sequences: one attention over the whole packed sequence with a block-
diagonal mask), (d) central finite differences, (e) limits: a window wider
than the sequence is no window, and tile liveness by brute force.
"""

import math

import numpy as np
import pytest
import torch

from oracle import (allowed_mask, attention_backward, attention_backward_varlen,
                    attention_forward, attention_forward_varlen, live_tiles)

RNG = np.random.default_rng(777)


def rand(*shape):
    return RNG.standard_normal(shape)


# ------------------------------------------------------------- (a) closed forms

def test_zero_window_is_the_diagonal():
    # window (0, 0): row i sees key i only -> O_i = V_i, LSE_i = scale q_i.k_i
    q, k, v = rand(2, 2, 9, 5), rand(2, 2, 9, 5), rand(2, 2, 9, 5)
    o, lse = attention_forward(q, k, v, 0.3, window=(0, 0))
    np.testing.assert_allclose(o, v, atol=1e-15, rtol=0)
    np.testing.assert_allclose(lse, 0.3 * np.sum(q * k, axis=-1), atol=1e-14, rtol=0)


def test_causal_window_of_one_is_two_key_softmax():
    # causal, window (1, .): row i sees keys i-1 and i
    n, d = 7, 3
    q, k, v = rand(1, 1, n, d), rand(1, 1, n, d), rand(1, 1, n, d)
    o, _ = attention_forward(q, k, v, 1.0, causal=True, window=(1, -1))
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15, rtol=0)
    for i in range(1, n):
        a = q[0, 0, i] @ k[0, 0, i - 1]
        b = q[0, 0, i] @ k[0, 0, i]
        w = 1.0 / (1.0 + math.exp(b - a))  # weight of key i-1
        np.testing.assert_allclose(o[0, 0, i], w * v[0, 0, i - 1] + (1 - w) * v[0, 0, i],
                                   atol=1e-14, rtol=0)


def test_wide_window_is_no_window():
    n = 20
    q, k, v = rand(1, 2, n, 4), rand(1, 2, n, 4), rand(1, 2, n, 4)
    for causal in (False, True):
        a = attention_forward(q, k, v, 0.5, causal=causal, window=(n, n))
        b = attention_forward(q, k, v, 0.5, causal=causal)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


# -------------------------------------------------------------- (b) brute force

@pytest.mark.parametrize("window", [(2, 1), (0, 3), (3, 0), (1, -1), (-1, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_window_brute_force(window, causal):
    n, d = 8, 3
    q, k, v = rand(1, 1, n, d), rand(1, 1, n, d), rand(1, 1, n, d)
    o, lse = attention_forward(q, k, v, 0.6, causal=causal, window=window)
    wl, wr = window
    for i in range(n):
        keys = [j for j in range(n) if (not causal or j <= i)
                and (wl < 0 or i - j <= wl) and (wr < 0 or j - i <= wr)]
        if not keys:
            assert np.isneginf(lse[0, 0, i]) and np.all(o[0, 0, i] == 0)
            continue
        w = [math.exp(0.6 * sum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(d))) for j in keys]
        z = sum(w)
        for c in range(d):
            want = sum(wi * v[0, 0, j, c] for wi, j in zip(w, keys)) / z
            assert abs(o[0, 0, i, c] - want) < 1e-12
        assert abs(lse[0, 0, i] - math.log(z)) < 1e-12


# ------------------------------------------------------ (c) library routines

def _sdpa(q, k, v, scale, ok):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.tensor(ok), scale=scale).numpy()


def _window_ok(n, causal, wl, wr):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    ok = np.ones((n, n), bool)
    if causal:
        ok &= j <= i
    if wl >= 0:
        ok &= j >= i - wl
    if wr >= 0:
        ok &= j <= i + wr
    return ok


@pytest.mark.parametrize("window,causal", [((5, 2), False), ((4, -1), True), ((0, 6), False)])
def test_window_against_sdpa_and_autograd(window, causal):
    n, d = 31, 6
    q, k, v, do = (rand(1, 2, n, d) for _ in range(4))
    ok = _window_ok(n, causal, *window)
    o, lse = attention_forward(q, k, v, 0.45, causal=causal, window=window)
    np.testing.assert_allclose(o[0], _sdpa(q[0], k[0], v[0], 0.45, ok), atol=1e-13, rtol=0)
    np.testing.assert_array_equal(allowed_mask(n, None, causal, window=window), ok)
    dq, dk, dv = attention_backward(q, k, v, do, 0.45, causal=causal, window=window)[:3]
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = (0.45 * qt @ kt.transpose(-1, -2)).masked_fill(~torch.tensor(ok), -math.inf)
    (torch.softmax(s, -1) @ vt * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12, rtol=0)


def _packed(lens, H, d):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    return cu, rand(T, H, d), rand(T, H, d), rand(T, H, d), rand(T, H, d)


@pytest.mark.parametrize("causal,window", [(False, None), (True, None), (True, (3, -1)),
                                           (False, (2, 2))])
def test_varlen_against_block_diagonal_sdpa(causal, window):
    lens = [5, 0, 13, 1, 9]
    H, d = 2, 4
    cu, q, k, v, do = _packed(lens, H, d)
    T = int(cu[-1])
    seq = np.repeat(np.arange(len(lens)), lens)
    pos = np.concatenate([np.arange(n) for n in lens])
    i, j = pos[:, None], pos[None, :]
    ok = seq[:, None] == seq[None, :]
    if causal:
        ok &= j <= i
    if window is not None:
        ok &= (j >= i - window[0]) & ((j <= i + window[1]) if window[1] >= 0 else True)
    o, lse = attention_forward_varlen(q, k, v, cu, 0.5, causal, window)
    qh, kh, vh = (np.transpose(x, (1, 0, 2)) for x in (q, k, v))
    ref = _sdpa(qh, kh, vh, 0.5, ok)
    np.testing.assert_allclose(np.transpose(o, (1, 0, 2)), ref, atol=1e-13, rtol=0)
    s = torch.tensor(0.5 * qh @ np.swapaxes(kh, -1, -2)).masked_fill(~torch.tensor(ok), -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-13, rtol=0)
    # gradients through torch autograd over the packed sequence
    dq, dk, dv = attention_backward_varlen(q, k, v, do, cu, 0.5, causal, window)[:3]
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (qh, kh, vh))
    sc = (0.5 * qt @ kt.transpose(-1, -2)).masked_fill(~torch.tensor(ok), -math.inf)
    (torch.softmax(sc, -1) @ vt * torch.tensor(np.transpose(do, (1, 0, 2)))).sum().backward()
    for got, t in ((dq, qt), (dk, kt), (dv, vt)):
        np.testing.assert_allclose(np.transpose(got, (1, 0, 2)), t.grad.numpy(), atol=1e-12, rtol=0)


# -------------------------------------------------- (d) finite differences

@pytest.mark.parametrize("window,causal", [((1, 1), False), ((2, -1), True)])
def test_window_gradients_central_differences(window, causal):
    rng = np.random.default_rng(5)
    n, d = 5, 3
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    grads = attention_backward(q, k, v, do, 0.7, causal=causal, window=window)[:3]

    def loss():
        return float(np.sum(attention_forward(q, k, v, 0.7, causal=causal, window=window)[0]
                            * do))

    for x, g in zip((q, k, v), grads):
        for idx in np.ndindex(x.shape):
            h = 1e-6 * max(1.0, abs(x[idx]))
            x0 = x[idx]
            x[idx] = x0 + h
            lp = loss()
            x[idx] = x0 - h
            lm = loss()
            x[idx] = x0
            assert abs((lp - lm) / (2 * h) - g[idx]) <= 1e-6 * max(1.0, abs(g[idx]))


# --------------------------------------------------- (e) tile liveness limits

@pytest.mark.parametrize("window,causal", [((100, 0), True), ((0, 0), False), ((300, 50), False),
                                           ((128, -1), True), ((-1, 130), False)])
def test_window_live_tiles_brute_force(window, causal):
    n, tile = 700, 128
    got = live_tiles(n, causal, window=window, tile=tile)
    ok = _window_ok(n, causal, *window)
    t = (n + tile - 1) // tile
    for qt in range(t):
        for kt in range(t):
            blk = ok[qt * tile:(qt + 1) * tile, kt * tile:(kt + 1) * tile]
            if blk.any():
                assert got[(qt, kt)] == int(not blk.all())
            else:
                assert (qt, kt) not in got
