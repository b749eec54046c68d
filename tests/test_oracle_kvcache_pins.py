"""Pins for the fp64 oracle of attention over a key/value cache and of the
merge of partial results.  CPU only.

The checks do not re-type the oracle's vectorised code: (a) brute force with
scalar loops on tiny inputs, (b) equivalence with the self-attention oracle
(pinned on its own in test_oracle_pins.py) on the equivalent full sequence,
(c) torch's scaled_dot_product_attention in fp64 with an explicit boolean
mask, (d) closed forms, and, for the merge, (e) the closed form
LSE = logsumexp_s LSE_s, O = sum_s e^{LSE_s - LSE} O_s through
torch.logsumexp, and exact identities (partition of the keys, order of the
parts, empty parts).
"""

import math

import numpy as np
import pytest
import torch

from oracle import (attention_forward, attention_forward_kvcache, kvcache_allowed,
                    merge_partial_states)

RNG = np.random.default_rng(4321)


def rand(*shape):
    return RNG.standard_normal(shape)


# ---------------------------------------------------------------- (a) brute force

def brute_kvcache(q, k, v, scale, causal, cache_len):
    """Scalar loops: for each row, list the keys the cache reading allows,
    sum e^{s} directly (inputs are small) and form the weighted mean of V."""
    B, H, nq, d = q.shape
    nk = k.shape[2]
    o = np.zeros((B, H, nq, v.shape[3]))
    lse = np.full((B, H, nq), -np.inf)
    for b in range(B):
        L = nk if cache_len is None else int(cache_len[b])
        for h in range(H):
            for r in range(nq):
                pos = L - nq + r  # absolute position of query row r
                keys = [j for j in range(min(L, nk)) if not causal or j <= pos]
                if not keys:
                    continue
                w = [math.exp(scale * sum(q[b, h, r, c] * k[b, h, j, c] for c in range(d)))
                     for j in keys]
                z = sum(w)
                for c in range(v.shape[3]):
                    o[b, h, r, c] = sum(wi * v[b, h, j, c] for wi, j in zip(w, keys)) / z
                lse[b, h, r] = math.log(z)
    return o, lse


@pytest.mark.parametrize("nq,nk,d", [(1, 1, 1), (1, 5, 3), (2, 4, 2), (3, 6, 3), (4, 3, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force(nq, nk, d, causal):
    q, k, v = rand(2, 2, nq, d), rand(2, 2, nk, d), rand(2, 2, nk, d)
    for cl in ([nk, nk], [max(nk - 1, 0), 1], [0, nk], [min(2, nk), max(nk - 2, 0)]):
        cache_len = np.array(cl, np.int32)
        o, lse = attention_forward_kvcache(q, k, v, 0.7, causal, cache_len)
        bo, blse = brute_kvcache(q, k, v, 0.7, causal, cache_len)
        np.testing.assert_allclose(o, bo, atol=1e-12)
        assert np.array_equal(np.isneginf(lse), np.isneginf(blse))
        fin = np.isfinite(blse)
        np.testing.assert_allclose(lse[fin], blse[fin], atol=1e-12)
        assert np.all(o[~fin] == 0.0)


def test_default_cache_len_is_all_slots():
    q, k, v = rand(1, 2, 3, 4), rand(1, 2, 9, 4), rand(1, 2, 9, 4)
    a = attention_forward_kvcache(q, k, v, 0.5, True)
    b = attention_forward_kvcache(q, k, v, 0.5, True, np.array([9]))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------- (b) self-attention equivalence

@pytest.mark.parametrize("causal", [False, True])
def test_rows_match_full_sequence_attention(causal):
    # The Nq query rows are the last Nq tokens of a length-L sequence: in a
    # full self-attention over that sequence (causal: j <= i; otherwise a key
    # padding of L) rows L-Nq .. L-1 give the same O and LSE.
    nq, nk, d = 5, 40, 6
    q, k, v = rand(2, 2, nq, d), rand(2, 2, nk, d), rand(2, 2, nk, d)
    cache_len = np.array([40, 23], np.int32)
    o, lse = attention_forward_kvcache(q, k, v, 0.3, causal, cache_len)
    for b in range(2):
        L = int(cache_len[b])
        qf = rand(1, 2, L, d)
        qf[0, :, L - nq:] = q[b]
        kv = None if causal else np.array([L], np.int32)
        of, lf = attention_forward(qf, k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.3,
                                   causal=causal, kv_len=kv)
        np.testing.assert_allclose(o[b], of[0, :, L - nq:], atol=1e-12)
        np.testing.assert_allclose(lse[b], lf[0, :, L - nq:], atol=1e-12)


def test_square_causal_is_plain_causal():
    n, d = 33, 8
    q, k, v = rand(1, 3, n, d), rand(1, 3, n, d), rand(1, 3, n, d)
    o, lse = attention_forward_kvcache(q, k, v, 0.25, True)
    of, lf = attention_forward(q, k, v, 0.25, causal=True)
    np.testing.assert_allclose(o, of, atol=1e-12)
    np.testing.assert_allclose(lse, lf, atol=1e-12)


# ------------------------------------------------------------- (c) torch SDPA

@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa(causal):
    nq, nk, d = 4, 50, 16
    q, k, v = rand(3, 2, nq, d), rand(3, 2, nk, d), rand(3, 2, nk, d)
    cache_len = np.array([50, 17, 4], np.int32)
    o, _ = attention_forward_kvcache(q, k, v, 0.25, causal, cache_len)
    for b in range(3):
        L = int(cache_len[b])
        pos = torch.arange(nq)[:, None] + (L - nq)
        j = torch.arange(nk)[None, :]
        m = ((j < L) & ((j <= pos) if causal else torch.ones_like(j, dtype=torch.bool)))
        m = m.expand(nq, nk)
        rows = m.any(dim=1).numpy()
        want = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[b]), torch.from_numpy(k[b]), torch.from_numpy(v[b]),
            attn_mask=m, scale=0.25).numpy()
        np.testing.assert_allclose(o[b][:, rows], want[:, rows], atol=1e-12)
        assert np.all(o[b][:, ~rows] == 0.0)


# ------------------------------------------------------------ (d) closed forms

def test_single_slot_returns_its_value():
    q, k, v = rand(2, 3, 2, 5), rand(2, 3, 7, 5), rand(2, 3, 7, 5)
    o, lse = attention_forward_kvcache(q, k, v, 0.9, False, np.array([1, 1]))
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :, :1], o.shape), atol=1e-15)
    np.testing.assert_allclose(lse, 0.9 * np.einsum("bhrc,bhc->bhr", q, k[:, :, 0]),
                               atol=1e-13)


def test_identical_keys_average_causal_prefix():
    # Equal keys: row r averages V over its allowed slots 0 .. L-Nq+r.
    nq, nk, d, L = 3, 12, 4, 10
    q, v = rand(1, 1, nq, d), rand(1, 1, nk, d)
    k = np.broadcast_to(rand(1, 1, 1, d), (1, 1, nk, d)).copy()
    o, lse = attention_forward_kvcache(q, k, v, 0.5, True, np.array([L]))
    for r in range(nq):
        cnt = L - nq + r + 1
        np.testing.assert_allclose(o[0, 0, r], v[0, 0, :cnt].mean(0), atol=1e-13)
        s = 0.5 * q[0, 0, r] @ k[0, 0, 0]
        assert abs(lse[0, 0, r] - (s + math.log(cnt))) < 1e-13


def test_rows_before_the_cache_start_are_empty():
    # Causal with Nq > L: rows at negative positions see no key.
    q, k, v = rand(1, 1, 4, 3), rand(1, 1, 6, 3), rand(1, 1, 6, 3)
    o, lse = attention_forward_kvcache(q, k, v, 1.0, True, np.array([2]))
    assert np.all(np.isneginf(lse[0, 0, :2])) and np.all(o[0, 0, :2] == 0)
    assert np.all(np.isfinite(lse[0, 0, 2:]))
    ok = kvcache_allowed(4, 6, 2, True)
    assert ok.sum(axis=1).tolist() == [0, 0, 1, 2]


# -------------------------------------------------------------------- (e) merge

def split_parts(q, k, v, scale, causal, cache_len, bounds):
    parts = [attention_forward_kvcache(q, k, v, scale, causal, cache_len, (lo, hi))
             for lo, hi in zip(bounds[:-1], bounds[1:])]
    return np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts])


@pytest.mark.parametrize("bounds", [[0, 64], [0, 20, 64], [0, 1, 2, 63, 64],
                                    [0, 16, 16, 32, 48, 64], [0, 30, 40, 50, 64]])
@pytest.mark.parametrize("causal", [False, True])
def test_merge_of_key_partition_is_whole(bounds, causal):
    nq, nk, d = 3, 64, 8
    q, k, v = rand(2, 2, nq, d), rand(2, 2, nk, d), rand(2, 2, nk, d)
    cache_len = np.array([64, 35], np.int32)
    whole = attention_forward_kvcache(q, k, v, 0.35, causal, cache_len)
    op, lp = split_parts(q, k, v, 0.35, causal, cache_len, bounds)
    o, lse = merge_partial_states(op, lp)
    np.testing.assert_allclose(o, whole[0], atol=1e-12)
    np.testing.assert_allclose(lse, whole[1], atol=1e-12)


def test_merge_matches_logsumexp_closed_form():
    S, R, d = 5, 40, 6
    op = rand(S, R, d)
    lp = 8.0 * rand(S, R)
    lp[1, :7] = -np.inf
    o, lse = merge_partial_states(op, lp)
    t = torch.from_numpy(lp)
    want_lse = torch.logsumexp(t, dim=0)
    w = torch.exp(t - want_lse).numpy()
    np.testing.assert_allclose(lse, want_lse.numpy(), atol=1e-12)
    np.testing.assert_allclose(o, np.einsum("sr,srd->rd", w, op), atol=1e-12)


def test_merge_order_and_identity():
    op, lp = rand(4, 10, 3), rand(4, 10)
    o, lse = merge_partial_states(op, lp)
    perm = [2, 0, 3, 1]
    o2, lse2 = merge_partial_states(op[perm], lp[perm])
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)
    o1, l1 = merge_partial_states(op[:1], lp[:1])
    np.testing.assert_allclose(o1, op[0], atol=1e-15)
    np.testing.assert_allclose(l1, lp[0], atol=1e-15)


def test_merge_equal_parts_and_empty_parts():
    op, lp = rand(2, 6, 4), rand(6)
    o, lse = merge_partial_states(op, np.stack([lp, lp]))
    np.testing.assert_allclose(o, 0.5 * (op[0] + op[1]), atol=1e-14)
    np.testing.assert_allclose(lse, lp + math.log(2.0), atol=1e-14)
    # parts with LSE = -inf contribute nothing; all-empty gives O = 0, -inf
    lp3 = np.stack([np.full(6, -np.inf), lp, np.full(6, -np.inf)])
    o3, l3 = merge_partial_states(np.concatenate([op[:1], op]), lp3)
    np.testing.assert_allclose(o3, op[0], atol=1e-15)
    np.testing.assert_allclose(l3, lp, atol=1e-15)
    oe, le = merge_partial_states(op, np.full((2, 6), -np.inf))
    assert np.all(oe == 0) and np.all(np.isneginf(le))


def test_merge_far_apart_parts_do_not_overflow():
    op = rand(2, 3, 4)
    lp = np.array([[1000.0, -1000.0, 5.0], [0.0, 0.0, 5.0 + 800.0]])
    o, lse = merge_partial_states(op, lp)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    np.testing.assert_allclose(o[0], op[0, 0], atol=1e-15)
    np.testing.assert_allclose(o[1], op[1, 1], atol=1e-15)
    np.testing.assert_allclose(o[2], op[1, 2], atol=1e-15)
    np.testing.assert_allclose(lse, [1000.0, 0.0, 805.0], atol=1e-12)
