"""Pins for the oracle's dropout: the Philox4x32-10 generator against the
known-answer vectors published with it (Random123 distribution, kat_vectors:
counter/key all zero, all ones, and the pi-digits vector), the statistics
of its bytes, and the dropout attention against (a) the undropped oracle at
p = 0, (b) torch autograd in fp64 with the keep mask as an explicit tensor,
(c) central finite differences (the mask is a fixed function of the seed),
(d) independence from the row chunking, (e) packed sequences by their
per-sequence head numbering.  CPU only."""

import math

import numpy as np
import pytest
import torch

from oracle import (attention_backward, attention_backward_varlen, attention_forward,
                    dropout_keep, dropout_p8, philox4x32_10)

RNG = np.random.default_rng(99)


def rand(*shape):
    return RNG.standard_normal(shape)


@pytest.mark.parametrize("ctr,key,want", [
    ((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff,) * 4, (0xffffffff,) * 2, (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
])
def test_philox_known_answers(ctr, key, want):
    got = philox4x32_10(*ctr, *key)
    assert tuple(int(x) for x in got) == want


def test_philox_vectorised_equals_elementwise():
    c0 = np.arange(50, dtype=np.uint64) * 7919
    vec = philox4x32_10(c0, 3, 5, 11, 0x1234, 0x9876)
    for t in range(50):
        one = philox4x32_10(int(c0[t]), 3, 5, 11, 0x1234, 0x9876)
        assert [int(x) for x in one] == [int(v[t]) for v in vec]


@pytest.mark.parametrize("p8", [26, 128, 230])
def test_keep_rate_and_byte_uniformity(p8):
    keep = dropout_keep(seed=2024, offset=3, p8=p8, bh=5, rows=np.arange(512),
                        cols=np.arange(2048))
    n = keep.size
    q = 1 - p8 / 256
    assert abs(keep.mean() - q) < 5 * math.sqrt(q * (1 - q) / n)
    # rows and column phases are not correlated with the keep bit
    assert np.abs(keep.mean(axis=1) - q).max() < 6 * math.sqrt(q * (1 - q) / 2048)
    for jj in range(16):
        assert abs(keep[:, jj::16].mean() - q) < 6 * math.sqrt(q * (1 - q) / (n / 16))


def test_seed_offset_and_head_change_the_mask():
    base = dropout_keep(7, 0, 128, 0, np.arange(64), np.arange(64))
    for other in (dropout_keep(8, 0, 128, 0, np.arange(64), np.arange(64)),
                  dropout_keep(7, 1, 128, 0, np.arange(64), np.arange(64)),
                  dropout_keep(7, 0, 128, 1, np.arange(64), np.arange(64))):
        assert 0.4 < (base != other).mean() < 0.6


def test_p8_rounding():
    assert dropout_p8(0.0) == 0 and dropout_p8(0.1) == 26 and dropout_p8(0.5) == 128
    assert dropout_p8(0.999) == 255
    with pytest.raises(ValueError):
        dropout_p8(1.0)


def test_zero_probability_is_no_dropout():
    q, k, v, do = (rand(1, 2, 40, 8) for _ in range(4))
    a = attention_backward(q, k, v, do, 0.3, causal=True, dropout=dict(p8=0, seed=1, offset=0))
    b = attention_backward(q, k, v, do, 0.3, causal=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_against_autograd_with_explicit_mask(causal):
    B, H, N, d = 2, 2, 37, 6
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    drop = dict(p8=77, seed=0x123456789, offset=5)
    dq, dk, dv, o, lse, _ = attention_backward(q, k, v, do, 0.4, causal=causal, dropout=drop)
    o2, lse2 = attention_forward(q, k, v, 0.4, causal=causal, dropout=drop)
    np.testing.assert_allclose(o, o2, atol=1e-13, rtol=0)
    for b in range(B):
        for h in range(H):
            z = dropout_keep(drop["seed"], drop["offset"], drop["p8"], b * H + h, np.arange(N),
                             np.arange(N)) / (1 - 77 / 256)
            qt, kt, vt = (torch.tensor(x[b, h], requires_grad=True) for x in (q, k, v))
            s = 0.4 * qt @ kt.T
            if causal:
                s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), -math.inf)
            p = torch.softmax(s, -1)
            ot = (p * torch.tensor(z)) @ vt
            np.testing.assert_allclose(o[b, h], ot.detach().numpy(), atol=1e-13, rtol=0)
            np.testing.assert_allclose(lse[b, h], torch.logsumexp(s, -1).detach().numpy(),
                                       atol=1e-13, rtol=0)
            (ot * torch.tensor(do[b, h])).sum().backward()
            np.testing.assert_allclose(dq[b, h], qt.grad.numpy(), atol=1e-12, rtol=0)
            np.testing.assert_allclose(dk[b, h], kt.grad.numpy(), atol=1e-12, rtol=0)
            np.testing.assert_allclose(dv[b, h], vt.grad.numpy(), atol=1e-12, rtol=0)


def test_dropout_gradients_central_differences():
    rng = np.random.default_rng(3)
    n, d = 6, 3
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    drop = dict(p8=100, seed=42, offset=0)
    grads = attention_backward(q, k, v, do, 0.9, causal=True, dropout=drop)[:3]

    def loss():
        return float(np.sum(attention_forward(q, k, v, 0.9, causal=True, dropout=drop)[0] * do))

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


def test_dropout_does_not_depend_on_row_chunking():
    q, k, v, do = (rand(1, 1, 50, 4) for _ in range(4))
    drop = dict(p8=60, seed=9, offset=1)
    a = attention_backward(q, k, v, do, 0.5, dropout=drop, row_chunk=7)
    b = attention_backward(q, k, v, do, 0.5, dropout=drop, row_chunk=1024)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13, rtol=0)


def test_single_head_slice_uses_its_global_head_index():
    q, k, v = (rand(2, 3, 20, 4) for _ in range(3))
    drop = dict(p8=90, seed=5, offset=0)
    full = attention_forward(q, k, v, 0.5, dropout=drop)[0]
    one = attention_forward(q[1:2, 2:3], k[1:2, 2:3], v[1:2, 2:3], 0.5,
                            dropout=dict(drop, bh0=1 * 3 + 2))[0]
    np.testing.assert_array_equal(full[1, 2], one[0, 0])


def test_packed_sequences_number_heads_per_sequence():
    lens = [9, 0, 14]
    H, d = 2, 3
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, do = (rand(T, H, d) for _ in range(4))
    drop = dict(p8=50, seed=11, offset=2)
    r = attention_backward_varlen(q, k, v, do, cu, 0.6, True, None, drop)
    for b, (lo, hi) in enumerate(zip(cu[:-1], cu[1:])):
        if hi == lo:
            continue
        sl = [np.transpose(x[lo:hi], (1, 0, 2))[None] for x in (q, k, v, do)]
        want = attention_backward(*sl, 0.6, causal=True, dropout=dict(drop, bh0=b * H))
        for got, w in zip(r[:4], want[:4]):
            np.testing.assert_array_equal(np.transpose(got[lo:hi], (1, 0, 2)), w[0])
