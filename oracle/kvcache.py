"""fp64 reference for attention over a key/value cache, and for merging
partial attention results computed over disjoint key sets.

TEST INFRASTRUCTURE ONLY: imported by tests, by the package smoke check and
by the benchmark's CPU-baseline leg, never by the product path.  It shares no
code with the CUDA library.

What it computes, and where the pages define it:

* Attention of a few new query rows against cached keys and values (page
  "FlashAttention", aiwiki, section "Software integration and limitations":
  the method's software offers inference with cached keys and values).  The
  arithmetic is the scaled dot-product formula of the same page, section
  "Attention and the memory bottleneck":
      S = scale * Q K^T,   P = softmax_row(S + mask),   O = P V
  with Q holding Nq rows and K, V holding the Nk cache slots of one head.
* Merging partial results (page "FlashAttention", aiwiki, section "Tiling
  and online normalization").  The running-max / running-sum / rescaled
  accumulator recurrence there folds in one score block at a time.  A
  partial result over a key subset, given as its normalised output O_s and
  log-sum-exp LSE_s, is the state (m = LSE_s, l = 1, u = O_s): both give
  the same u / l and m + ln l.  Folding such states into the running state
  with the same three update rules gives the result over the union of the
  key subsets:
      m' = max(m, m_s)
      l' = e^{m - m'} l + e^{m_s - m'}
      u' = e^{m - m'} u + e^{m_s - m'} O_s
      O  = u / l,   LSE = m + ln l

Readings where the pages are silent (each is listed in the design notes):
* Cache length.  cache_len[b] (default Nk) is the number of valid cache
  slots of batch element b; slots j >= cache_len[b] are never attended.
* Query positions.  The Nq query rows are the last Nq tokens of the
  sequence held in the cache: row r sits at position cache_len[b] - Nq + r.
  With ``causal`` row r may attend key j only if j <= cache_len[b] - Nq + r
  (so with Nq = Nk = cache_len this is the usual causal mask j <= i).
* A row with no allowed key has O = 0 and LSE = -inf, as in the main
  oracle; in a merge, a part with LSE = -inf contributes nothing, and a
  merge of only such parts gives O = 0, LSE = -inf.
"""

import numpy as np


def kvcache_allowed(nq, nk, cache_len, causal=False, key_range=None):
    """Boolean [nq, nk]: which (query row, cache slot) pairs may interact.

    ``key_range`` = (lo, hi) further restricts the keys to lo <= j < hi (the
    key subset of one partial result).
    """
    r = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    ok = np.broadcast_to(j < cache_len, (nq, nk)).copy()
    if causal:
        ok &= j <= cache_len - nq + r
    if key_range is not None:
        lo, hi = key_range
        ok &= (j >= lo) & (j < hi)
    return ok


def attention_forward_kvcache(q, k, v, scale, causal=False, cache_len=None,
                              key_range=None):
    """O [B,H,Nq,d] and LSE [B,H,Nq] of Nq query rows against an Nk-slot cache.

    q: [B,H,Nq,d]; k, v: [B,H,Nk,d]; cache_len: int [B] or None (= Nk).
    Two-pass softmax over the allowed keys of each row, in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, nq, _ = q.shape
    nk = k.shape[2]
    o = np.zeros((B, H, nq, v.shape[3]))
    lse = np.full((B, H, nq), -np.inf)
    for b in range(B):
        L = nk if cache_len is None else min(max(int(cache_len[b]), 0), nk)
        ok = kvcache_allowed(nq, nk, L, causal, key_range)
        for h in range(H):
            s = np.where(ok, scale * (q[b, h] @ k[b, h].T), -np.inf)
            m = s.max(axis=1)
            live = np.isfinite(m)
            m0 = np.where(live, m, 0.0)
            e = np.where(ok, np.exp(s - m0[:, None]), 0.0)
            l = e.sum(axis=1)
            l1 = np.where(live, l, 1.0)
            o[b, h] = (e / l1[:, None]) @ v[b, h]
            lse[b, h] = np.where(live, m0 + np.log(l1), -np.inf)
    return o, lse


def merge_partial_states(o_parts, lse_parts):
    """Merge S partial results over disjoint key sets into one.

    o_parts: [S, ..., d] normalised partial outputs; lse_parts: [S, ...]
    their log-sum-exps (natural log, -inf for an empty part).  Returns
    (O [..., d], LSE [...]).  Folds the parts in order into the running
    state (m, l, u) by the online-normalisation update rules.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.full(lse_parts.shape[1:], -np.inf)
    l = np.zeros(lse_parts.shape[1:])
    u = np.zeros(o_parts.shape[1:])
    for o_s, m_s in zip(o_parts, lse_parts):
        m_new = np.maximum(m, m_s)
        fin = np.isfinite(m_new)
        ref = np.where(fin, m_new, 0.0)
        a_old = np.where(np.isfinite(m), np.exp(m - ref), 0.0)
        a_new = np.where(np.isfinite(m_s), np.exp(m_s - ref), 0.0)
        l = a_old * l + a_new
        u = a_old[..., None] * u + a_new[..., None] * o_s
        m = m_new
    live = l > 0
    l1 = np.where(live, l, 1.0)
    o = np.where(live[..., None], u / l1[..., None], 0.0)
    lse = np.where(live, m + np.log(l1), -np.inf)
    return o, lse
