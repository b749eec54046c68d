"""Pins for the fp64 oracle: closed forms, library routines, calculus and
invariants that the oracle must reproduce.  CPU only.

Each test names the fact it relies on.  None re-types the oracle's own
vectorised code: the checks are (a) closed forms of attention on special
inputs, (b) an independent library implementation (torch SDPA and torch
autograd, fp64 CPU), (c) central finite differences, (d) exact invariants
of softmax attention, (e) slicing equivalences for the masks, and (f) the
tiled online recurrence (page "FlashAttention", aiwiki, "Tiling and online
normalization") against the two-pass definition.
"""

import math

import numpy as np
import pytest
import torch

from oracle import (allowed_mask, attention_backward, attention_forward,
                    attention_forward_online, attention_forward_rows,
                    live_tiles)

RNG = np.random.default_rng(1234)


def rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- (a) closed forms

@pytest.mark.parametrize("d", [1, 4, 64])
def test_single_key_output_is_value(d):
    # N = 1: softmax over one key is 1, so O = V and LSE = the one score.
    q, k, v = rand(2, 3, 1, d), rand(2, 3, 1, d), rand(2, 3, 1, d)
    o, lse = attention_forward(q, k, v, 0.37)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.37 * np.sum(q * k, axis=-1), atol=1e-14)


@pytest.mark.parametrize("n,kv", [(7, None), (9, 4), (130, 70)])
def test_identical_keys_average_values(n, kv):
    # Equal keys give equal scores along a row: P is uniform over the allowed
    # keys, O is their mean, LSE = s + ln(count), and dQ = 0 because every
    # dS row is P * (dP - sum_j P dP), whose product with identical keys
    # vanishes.
    d = 5
    q, v, do = rand(1, 1, n, d), rand(1, 1, n, d), rand(1, 1, n, d)
    k = np.broadcast_to(rand(1, 1, 1, d), (1, 1, n, d)).copy()
    kvl = None if kv is None else np.array([kv], np.int32)
    o, lse = attention_forward(q, k, v, 0.5, kv_len=kvl)
    cnt = n if kv is None else kv
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, :cnt].mean(0), (n, d)),
                               atol=1e-13)
    s = 0.5 * q[0, 0] @ k[0, 0, 0]
    np.testing.assert_allclose(lse[0, 0], s + math.log(cnt), atol=1e-13)
    dq = attention_backward(q, k, v, do, 0.5, kv_len=kvl)[0]
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)


def test_causal_identical_keys_prefix_mean():
    # Causal + equal keys: row i averages V[0..i].
    n, d = 11, 3
    q, v = rand(1, 1, n, d), rand(1, 1, n, d)
    k = np.ones((1, 1, n, d))
    o, lse = attention_forward(q, k, v, 1.0, causal=True)
    want = np.cumsum(v[0, 0], axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], want, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], q[0, 0].sum(1) + np.log(np.arange(1, n + 1)),
                               atol=1e-13)


def test_dominant_logit_selects_row():
    # One score exceeding the others by 60 gives P within e^-60 of one-hot.
    n, d = 16, 8
    q = np.zeros((1, 1, n, d))
    k = np.zeros((1, 1, n, d))
    v = rand(1, 1, n, d)
    q[0, 0, :, 0] = 1.0
    k[0, 0, 5, 0] = 60.0
    o, _ = attention_forward(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, 5], (n, d)),
                               atol=n * math.exp(-60) * np.abs(v).max() + 1e-15)


def test_causal_first_row_is_first_value():
    q, k, v = rand(2, 2, 9, 4), rand(2, 2, 9, 4), rand(2, 2, 9, 4)
    o, lse = attention_forward(q, k, v, 0.3, causal=True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.sum(q[:, :, 0] * k[:, :, 0], -1),
                               atol=1e-14)


def test_two_keys_closed_form():
    # N = 2, d = 1, no mask: P_i0 = 1 / (1 + e^{s_i1 - s_i0}), written out.
    q = np.array([0.3, -1.2]).reshape(1, 1, 2, 1)
    k = np.array([0.7, 2.0]).reshape(1, 1, 2, 1)
    v = np.array([1.5, -0.5]).reshape(1, 1, 2, 1)
    o, lse = attention_forward(q, k, v, 1.0)
    for i, qi in enumerate([0.3, -1.2]):
        s0, s1 = qi * 0.7, qi * 2.0
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))
        assert abs(o[0, 0, i, 0] - (p0 * 1.5 + (1 - p0) * -0.5)) < 1e-15
        assert abs(lse[0, 0, i] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14


def test_fully_masked_row_is_zero_and_inert():
    # Reading: a query row with no allowed key outputs 0, LSE = -inf, dQ = 0,
    # and adds nothing to dK / dV.
    n, d = 6, 3
    q, k, v, do = (rand(1, 1, n, d) for _ in range(4))
    kvl = np.array([0], np.int32)
    o, lse = attention_forward(q, k, v, 1.0, kv_len=kvl)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))
    dq, dk, dv = attention_backward(q, k, v, do, 1.0, kv_len=kvl)[:3]
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


# ------------------------------------------------ (b) independent library routines

def _torch_attention(q, k, v, scale, ok):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v))
    m = torch.tensor(ok)
    return torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=m, scale=scale).numpy()


@pytest.mark.parametrize("mask", ["none", "causal", "kv_len", "block"])
def test_forward_matches_torch_sdpa_fp64(mask):
    B, H, N, d, tile = 2, 3, 37, 8, 8
    q, k, v = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
    causal = mask == "causal"
    kv = np.array([20, 37], np.int32) if mask == "kv_len" else None
    t = (N + tile - 1) // tile
    bm = None
    if mask == "block":
        bm = (RNG.random((t, t)) < 0.5).astype(np.uint8)
        np.fill_diagonal(bm, 1)  # every row keeps a tile: no NaN rows in SDPA
    o, lse = attention_forward(q, k, v, 0.21, causal, bm, kv, tile=tile)
    for b in range(B):
        ok = allowed_mask(N, None, causal, bm, None if kv is None else kv[b], tile)
        ref = _torch_attention(q[b], k[b], v[b], 0.21, ok)
        np.testing.assert_allclose(o[b], ref, atol=1e-13, rtol=0)
        s = torch.tensor(0.21 * q[b] @ np.swapaxes(k[b], -1, -2))
        s = s.masked_fill(~torch.tensor(ok), -math.inf)
        np.testing.assert_allclose(lse[b], torch.logsumexp(s, -1).numpy(), atol=1e-13)


@pytest.mark.parametrize("mask", ["none", "causal", "kv_len", "block"])
def test_backward_matches_torch_autograd_fp64(mask):
    B, H, N, d, tile = 1, 2, 29, 6, 4
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    causal = mask == "causal"
    kv = np.array([17], np.int32) if mask == "kv_len" else None
    t = (N + tile - 1) // tile
    bm = None
    if mask == "block":
        bm = (RNG.random((t, t)) < 0.4).astype(np.uint8)
        np.fill_diagonal(bm, 1)
    dq, dk, dv = attention_backward(q, k, v, do, 0.4, causal, bm, kv, tile=tile)[:3]
    ok = torch.tensor(allowed_mask(N, None, causal, bm,
                                   None if kv is None else kv[0], tile))
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = (0.4 * qt @ kt.transpose(-1, -2)).masked_fill(~ok, -math.inf)
    o = torch.softmax(s, -1) @ vt
    (o * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


# ------------------------------------------------------ (c) finite differences

def _loss(q, k, v, do, scale, **kw):
    return float(np.sum(attention_forward(q, k, v, scale, **kw)[0] * do))


@pytest.mark.parametrize("n,d", [(3, 2), (5, 4)])
@pytest.mark.parametrize("mask", ["none", "causal", "kv_len", "block"])
def test_gradients_match_central_differences(n, d, mask):
    rng = np.random.default_rng(n * 10 + d)
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    kw = dict(causal=mask == "causal", tile=2)
    if mask == "kv_len":
        kw["kv_len"] = np.array([n - 1], np.int32)
    if mask == "block":
        t = (n + 1) // 2
        bm = np.ones((t, t), np.uint8)
        bm[0, -1] = 0
        kw["block_mask"] = bm
    scale = 0.8
    grads = attention_backward(q, k, v, do, scale, **kw)[:3]
    for x, g in zip((q, k, v), grads):
        for idx in np.ndindex(x.shape):
            h = 1e-6 * max(1.0, abs(x[idx]))
            x0 = x[idx]
            x[idx] = x0 + h
            lp = _loss(q, k, v, do, scale, **kw)
            x[idx] = x0 - h
            lm = _loss(q, k, v, do, scale, **kw)
            x[idx] = x0
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (idx, fd, g[idx])


# ------------------------------------------------------------- (d) invariants

@pytest.mark.parametrize("mask", ["none", "causal", "kv_len"])
def test_gradient_invariants(mask):
    # sum_j dS_ij = 0 for every row => sum_j dK_j = 0;
    # sum_j P_ij = 1 on live rows   => sum_j dV_j = sum over live rows of dO_i.
    B, H, N, d = 2, 2, 50, 7
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    kv = np.array([13, 50], np.int32) if mask == "kv_len" else None
    dq, dk, dv, o, lse, D = attention_backward(q, k, v, do, 0.3, mask == "causal",
                                               None, kv)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(D, np.sum(o * do, -1), atol=1e-13)


def test_key_value_joint_permutation_invariance():
    q, k, v = rand(1, 2, 33, 5), rand(1, 2, 33, 5), rand(1, 2, 33, 5)
    perm = RNG.permutation(33)
    o1, l1 = attention_forward(q, k, v, 0.6)
    o2, l2 = attention_forward(q, k[:, :, perm], v[:, :, perm], 0.6)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_row_chunking_does_not_change_result():
    q, k, v, do = (rand(1, 1, 70, 4) for _ in range(4))
    a = attention_backward(q, k, v, do, 0.5, True, row_chunk=1024)
    b = attention_backward(q, k, v, do, 0.5, True, row_chunk=9)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13)


# ------------------------------------------------------- (e) mask equivalences

def test_key_padding_equals_truncated_keys():
    # Keys j >= kv_len take no part: same as attention over K[:L], V[:L].
    N, d, L = 40, 6, 23
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    o, lse = attention_forward(q, k, v, 0.7, kv_len=np.array([L], np.int32))
    s = 0.7 * q[0, 0] @ k[0, 0, :L].T
    p = np.exp(s - s.max(1, keepdims=True))
    np.testing.assert_allclose(o[0, 0], (p / p.sum(1, keepdims=True)) @ v[0, 0, :L],
                               atol=1e-13)


def test_block_mask_equals_gathered_keys():
    # Row i attends exactly to the keys of its allowed tiles.
    N, d, tile = 24, 3, 4
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    t = N // tile
    bm = (RNG.random((t, t)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    o, _ = attention_forward(q, k, v, 1.0, block_mask=bm, tile=tile)
    for i in range(N):
        keys = [j for j in range(N) if bm[i // tile, j // tile]]
        s = q[0, 0, i] @ k[0, 0, keys].T
        p = np.exp(s - s.max())
        np.testing.assert_allclose(o[0, 0, i], (p / p.sum()) @ v[0, 0, keys], atol=1e-13)


def test_all_ones_block_mask_equals_dense():
    q, k, v = rand(1, 2, 19, 4), rand(1, 2, 19, 4), rand(1, 2, 19, 4)
    a = attention_forward(q, k, v, 0.5)
    b = attention_forward(q, k, v, 0.5, block_mask=np.ones((5, 5), np.uint8), tile=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_causal_equals_explicit_lower_triangle():
    N = 21
    q, k, v = rand(1, 1, N, 3), rand(1, 1, N, 3), rand(1, 1, N, 3)
    o, _ = attention_forward(q, k, v, 1.0, causal=True)
    ref = _torch_attention(q[0], k[0], v[0], 1.0, np.tril(np.ones((N, N), bool)))
    np.testing.assert_allclose(o[0], ref, atol=1e-13)


def test_sampled_rows_match_full_forward():
    q, k, v = rand(2, 2, 45, 4), rand(2, 2, 45, 4), rand(2, 2, 45, 4)
    kv = np.array([30, 45], np.int32)
    o, lse = attention_forward(q, k, v, 0.5, True, None, kv)
    rows = np.array([0, 7, 29, 44])
    for b in range(2):
        orow, lrow = attention_forward_rows(q, k, v, 0.5, b, 1, rows, True, None, kv)
        np.testing.assert_allclose(orow, o[b, 1, rows], atol=1e-14)
        np.testing.assert_allclose(lrow, lse[b, 1, rows], atol=1e-14)


# --------------------------------------------------- (f) online recurrence

@pytest.mark.parametrize("bq,bk", [(1, 1), (3, 5), (16, 16), (128, 7), (128, 128)])
@pytest.mark.parametrize("mask", ["none", "causal", "kv_len", "block"])
def test_online_recurrence_equals_two_pass(bq, bk, mask):
    B, H, N, d, tile = 1, 2, 37, 5, 8
    q, k, v = rand(B, H, N, d) * 3, rand(B, H, N, d) * 3, rand(B, H, N, d)
    kw = dict(causal=mask == "causal", tile=tile)
    if mask == "kv_len":
        kw["kv_len"] = np.array([11], np.int32)
    if mask == "block":
        t = (N + tile - 1) // tile
        bm = (RNG.random((t, t)) < 0.5).astype(np.uint8)
        bm[1, :] = 0  # a fully masked row block
        kw["block_mask"] = bm
    o1, l1 = attention_forward(q, k, v, 0.9, **kw)
    o2, l2 = attention_forward_online(q, k, v, 0.9, block_q=bq, block_k=bk, **kw)
    scale_o = max(1.0, np.abs(o1).max())
    assert np.abs(o1 - o2).max() <= 1e-12 * scale_o
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    assert np.abs(l1[fin] - l2[fin]).max() <= 1e-12 * max(1.0, np.abs(l1[fin]).max())


# ------------------------------------------------------- tile enumeration

def test_live_tiles_causal_closed_form():
    # Causal with N a multiple of the tile: T(T+1)/2 live tiles, only the T
    # diagonal ones partial.
    t = 8
    lt = live_tiles(t * 128, causal=True)
    assert len(lt) == t * (t + 1) // 2
    assert sorted(k for k, f in lt.items() if f) == [(i, i) for i in range(t)]


def test_live_tiles_band_global_count():
    # 128 tiles, band |i-j|<=1 (382 tiles) united with 8 global columns
    # (1024 tiles), overlap 2 + 7*3 = 23: 1383 live, none partial.
    from exact_io_aware_tma_gb300.workloads import band_global_block_mask
    bm = band_global_block_mask(128)
    assert int(bm.sum()) == 1383
    lt = live_tiles(256, block_mask=bm[:2, :2])
    assert lt == {(0, 0): 0, (0, 1): 0, (1, 0): 0, (1, 1): 0}


def test_live_tiles_key_padding():
    # kv_len = 300 over N = 512: key tiles 0, 1 full, tile 2 partial, 3 dead.
    lt = live_tiles(512, kv_len=300)
    assert lt == {(qt, kt): int(kt == 2) for qt in range(4) for kt in range(3)}
