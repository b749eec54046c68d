"""Plain, slow, fp64 reference for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY: imported by tests, by the package smoke check and
by the benchmark's CPU-baseline leg, never by the product path.  It shares no
code with the CUDA library.

What it computes, and where the pages define it:

* Forward (page "FlashAttention", aiwiki, section "Attention and the memory
  bottleneck", the displayed SDPA formula):
      S = scale * Q K^T,   P = softmax_row(S + mask),   O = P V
  Masks "restrict permitted query-key interactions" (same section); here a
  disallowed pair gets S = -inf before the softmax.
* Stored row statistic: the per-row log-sum-exp LSE_i = m_i + ln l_i of the
  scaled, masked scores (page "FlashAttention IO-aware explained", section
  "Recomputation and IO complexity": compact row statistics (m, l) kept for
  the backward pass; page "Fast and Memory Efficient Exact Attention",
  "Summary & Methodology Analysis": the softmax normalisation factor is
  stored).  LSE is the natural log.
* Backward: the exact gradient of L = sum(O * dO) with respect to Q, K, V,
  written out by calculus on the forward formula (the pages defer the
  closed form to the paper's appendices B.2/B.4, page "FlashAttention: Fast
  and Memory-Efficient Exact Attention with IO-Awareness", claims on
  "B.2 Memory-efficient backward pass"):
      dV = P^T dO
      dP = dO V^T
      D_i = sum_c dO_ic O_ic          (= sum_j P_ij dP_ij)
      dS = P * (dP - D)
      dQ = scale * dS K,   dK = scale * dS^T Q
* Online (tiled) forward, used only as a self-check of the two-pass path:
  the running-max / running-sum / rescaled-accumulator recurrence of page
  "FlashAttention" (aiwiki), section "Tiling and online normalization":
      m' = max(m, max s_b)
      l' = e^{m - m'} l + sum_j e^{s_bj - m'}
      u' = e^{m - m'} u + sum_j e^{s_bj - m'} v_bj
      O  = u / l
* Block-sparse masking: a predefined mask over 128x128 tiles; a pair (i, j)
  is allowed only if its tile is nonzero (page "Fast and Memory Efficient
  Exact Attention", "Summary & Methodology Analysis": zero blocks of a
  predefined block-sparsity mask are skipped).
* Dropout on the attention probabilities (page "FlashAttention: Fast and
  Memory-Efficient Exact Attention with IO-Awareness", claims on the
  backward pass: the dropout mask is not stored but regenerated from the
  generator state in the backward).  Reading: inverted dropout of P,
      O = ((P o Z) / (1 - p)) V,   Z_ij = keep bit of (b, h, i, j),
  LSE unchanged; backward dV = ((P o Z)/(1-p))^T dO, dP = (dO V^T) o Z/(1-p),
  D_i = sum_c dO_ic O_ic (still equal to sum_j P_ij dP_ij), dS = P o (dP - D).
  Z comes from oracle/philox.py (Philox4x32-10, element mapping there).
* Sliding-window masks and variable-length sequences (page "FlashAttention",
  aiwiki, section "Software integration and limitations": the method's
  software offers causal and sliding-window masks and variable-length
  sequences).  The pages give no formula for either; the readings below are
  the plain ones.

Readings where the pages are silent (each is listed in the design notes):
* allowed(b, i, j) = (not causal or j <= i)
                     and (block_mask is None or block_mask[i//128][j//128] != 0)
                     and (kv_len is None or j < kv_len[b])
                     and (window_left is None or j >= i - window_left)
                     and (window_right is None or j <= i + window_right).
  A window of (w, 0) with causal is the usual causal sliding window: query i
  sees keys i-w .. i.
* Variable-length sequences come packed: Q, K, V of shape [T, H, d] hold the
  B sequences back to back, sequence b being rows cu_seqlens[b] ..
  cu_seqlens[b+1]-1; each sequence attends only within itself, as a batch
  element of length cu_seqlens[b+1] - cu_seqlens[b] would.
* A row with no allowed key has O_i = 0, LSE_i = -inf and contributes no
  gradient.
* Inputs are whatever arrays the caller passes (the tests pass the bf16
  values the GPU receives, upcast to fp64); all arithmetic here is fp64.
"""

import numpy as np

from .philox import dropout_keep

TILE = 128  # side of one block-mask tile, in queries and in keys


def allowed_mask(n, rows=None, causal=False, block_mask=None, kv_len=None,
                 tile=TILE, window=None):
    """Boolean [len(rows), n]: which (query row, key column) pairs may interact.

    ``kv_len`` is the scalar valid-key count of ONE batch element (or None);
    ``window`` = (left, right), either bound None (or negative) = unbounded.
    """
    rows = np.arange(n) if rows is None else np.asarray(rows)
    cols = np.arange(n)
    ok = np.ones((rows.shape[0], n), dtype=bool)
    if causal:
        ok &= cols[None, :] <= rows[:, None]
    if window is not None:
        left, right = window
        if left is not None and left >= 0:
            ok &= cols[None, :] >= rows[:, None] - left
        if right is not None and right >= 0:
            ok &= cols[None, :] <= rows[:, None] + right
    if block_mask is not None:
        bm = np.asarray(block_mask)
        ok &= bm[rows[:, None] // tile, cols[None, :] // tile] != 0
    if kv_len is not None:
        ok &= cols[None, :] < int(kv_len)
    return ok


def _softmax_rows(s, ok):
    """Two-pass masked softmax of score rows: returns (P, LSE)."""
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1)
    live = np.isfinite(m)
    m0 = np.where(live, m, 0.0)
    e = np.where(ok, np.exp(s - m0[:, None]), 0.0)
    l = e.sum(axis=1)
    l1 = np.where(live, l, 1.0)
    p = e / l1[:, None]
    lse = np.where(live, m0 + np.log(l1), -np.inf)
    return p, lse


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _dropout_factor(dropout, bh, rows, n):
    """Z / (1 - p) for the given rows of head bh (None when no dropout).

    ``dropout`` = dict(p8=, seed=, offset=, bh0=0): the global head index of
    local head (b, h) is bh0 + b*H + h (a caller passing one sliced head
    passes its global index as bh0).
    """
    if dropout is None or dropout["p8"] == 0:
        return None
    keep = dropout_keep(dropout["seed"], dropout["offset"], dropout["p8"], bh, rows,
                        np.arange(n))
    return keep / (1.0 - dropout["p8"] / 256.0)


def _kv(kv_len, b):
    return None if kv_len is None else int(np.asarray(kv_len)[b])


def attention_forward(q, k, v, scale, causal=False, block_mask=None,
                      kv_len=None, heads=None, row_chunk=1024, tile=TILE,
                      window=None, dropout=None):
    """O [B,H,N,dv] and LSE [B,H,N] by the textbook two-pass definition.

    ``heads`` optionally restricts the work to a list of (b, h) pairs; the
    other heads of the result are left as NaN.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, _ = q.shape
    o = np.full(v.shape[:3] + (v.shape[3],), np.nan)
    lse = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else
                 [(b, h) for b in range(B) for h in range(H)]):
        for r0 in range(0, N, row_chunk):
            rows = np.arange(r0, min(N, r0 + row_chunk))
            s = scale * (q[b, h, rows] @ k[b, h].T)
            ok = allowed_mask(N, rows, causal, block_mask, _kv(kv_len, b),
                              tile, window)
            p, lse[b, h, rows] = _softmax_rows(s, ok)
            z = _dropout_factor(dropout, (dropout or {}).get("bh0", 0) + b * H + h, rows, N)
            o[b, h, rows] = (p if z is None else p * z) @ v[b, h]
    return o, lse


def attention_forward_rows(q, k, v, scale, b, h, rows, causal=False,
                           block_mask=None, kv_len=None, tile=TILE, window=None):
    """O and LSE of selected query rows of one head (sampled full-size checks)."""
    q, k, v = _as64(q[b, h]), _as64(k[b, h]), _as64(v[b, h])
    rows = np.asarray(rows)
    s = scale * (q[rows] @ k.T)
    ok = allowed_mask(k.shape[0], rows, causal, block_mask, _kv(kv_len, b),
                      tile, window)
    p, lse = _softmax_rows(s, ok)
    return p @ v, lse


def attention_backward(q, k, v, do, scale, causal=False, block_mask=None,
                       kv_len=None, heads=None, row_chunk=1024, tile=TILE,
                       window=None, dropout=None):
    """dQ, dK, dV [B,H,N,d] of L = sum(O * dO), plus O, LSE and D.

    P is rebuilt here from the inputs (the oracle stores nothing between
    passes); D uses this function's own fp64 O.  Returns
    (dq, dk, dv, o, lse, D).
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, _ = q.shape
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    o = np.full(v.shape, np.nan)
    lse = np.full((B, H, N), np.nan)
    dd = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else
                 [(b, h) for b in range(B) for h in range(H)]):
        dk[b, h] = 0.0
        dv[b, h] = 0.0
        for r0 in range(0, N, row_chunk):
            rows = np.arange(r0, min(N, r0 + row_chunk))
            s = scale * (q[b, h, rows] @ k[b, h].T)
            ok = allowed_mask(N, rows, causal, block_mask, _kv(kv_len, b),
                              tile, window)
            p, lse[b, h, rows] = _softmax_rows(s, ok)
            z = _dropout_factor(dropout, (dropout or {}).get("bh0", 0) + b * H + h, rows, N)
            pz = p if z is None else p * z
            o_r = pz @ v[b, h]
            o[b, h, rows] = o_r
            d_r = np.sum(do[b, h, rows] * o_r, axis=1)
            dd[b, h, rows] = d_r
            dp = do[b, h, rows] @ v[b, h].T
            if z is not None:
                dp = dp * z
            ds = p * (dp - d_r[:, None])
            dq[b, h, rows] = scale * (ds @ k[b, h])
            dk[b, h] += scale * (ds.T @ q[b, h, rows])
            dv[b, h] += pz.T @ do[b, h, rows]
    return dq, dk, dv, o, lse, dd


def attention_forward_online(q, k, v, scale, causal=False, block_mask=None,
                             kv_len=None, block_q=128, block_k=128, tile=TILE,
                             window=None):
    """O and LSE by the tiled online-softmax recurrence (self-check path).

    Visits query blocks of ``block_q`` rows and, for each, key blocks of
    ``block_k`` columns in order, carrying (m, l, u) per row exactly as the
    recurrence states; never forms a full score row.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, _ = q.shape
    o = np.zeros(v.shape)
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, block_q):
                rows = np.arange(r0, min(N, r0 + block_q))
                m = np.full(rows.shape[0], -np.inf)
                l = np.zeros(rows.shape[0])
                u = np.zeros((rows.shape[0], v.shape[3]))
                for c0 in range(0, N, block_k):
                    cols = np.arange(c0, min(N, c0 + block_k))
                    s_b = scale * (q[b, h, rows] @ k[b, h, cols].T)
                    ok = allowed_mask(N, rows, causal, block_mask,
                                      _kv(kv_len, b), tile, window)[:, cols]
                    s_b = np.where(ok, s_b, -np.inf)
                    m_new = np.maximum(m, s_b.max(axis=1))
                    # e^{m - m'}: 0 when nothing was seen yet (m = -inf);
                    # rows still without an allowed key keep l = 0, u = 0.
                    fin = np.isfinite(m_new)
                    ref = np.where(fin, m_new, 0.0)
                    alpha = np.where(np.isfinite(m), np.exp(m - ref), 0.0)
                    e = np.where(ok, np.exp(s_b - ref[:, None]), 0.0)
                    l = alpha * l + e.sum(axis=1)
                    u = alpha[:, None] * u + e @ v[b, h, cols]
                    m = m_new
                live = l > 0
                o[b, h, rows] = np.where(live[:, None],
                                         u / np.where(live, l, 1.0)[:, None],
                                         0.0)
                lse[b, h, rows] = np.where(
                    live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    return o, lse


def live_tiles(n, causal=False, block_mask=None, kv_len=None, tile=TILE,
               window=None):
    """Live (query tile, key tile) pairs of one batch element, by brute force.

    A tile pair is live when at least one of its (i, j) pairs is allowed; it
    is "partial" when it is live but not every one of its in-range pairs is
    allowed.  Returns a dict {(qt, kt): partial_flag} -- the enumeration the
    tiled kernels must visit (tiles with no allowed pair are skipped).
    """
    t = (n + tile - 1) // tile
    ok = allowed_mask(n, None, causal, block_mask, kv_len, tile, window)
    out = {}
    for qt in range(t):
        r = slice(qt * tile, min(n, (qt + 1) * tile))
        for kt in range(t):
            c = slice(kt * tile, min(n, (kt + 1) * tile))
            blk = ok[r, c]
            if blk.any():
                out[(qt, kt)] = int(not blk.all())
    return out


def _seq_dropout(dropout, b, H):
    """Dropout of packed sequence b: its heads are global heads b*H + h."""
    return None if dropout is None else dict(dropout, bh0=b * H)


def _varlen_heads(x, cu_seqlens, b):
    """Rows of sequence b of a packed [T, H, d] array, as a [1, H, len, d] view."""
    lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
    return np.transpose(_as64(x)[lo:hi], (1, 0, 2))[None]


def attention_forward_varlen(q, k, v, cu_seqlens, scale, causal=False,
                             window=None, dropout=None):
    """O [T,H,d] and LSE [H,T] of packed variable-length sequences: every
    sequence b (rows cu_seqlens[b] .. cu_seqlens[b+1]-1) attends within
    itself by the same definition as a batch element of its own length."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    T, H, _ = q.shape
    o = np.zeros(v.shape)
    lse = np.full((H, T), -np.inf)
    for b in range(len(cu_seqlens) - 1):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if hi <= lo:
            continue
        ob, lb = attention_forward(_varlen_heads(q, cu_seqlens, b),
                                   _varlen_heads(k, cu_seqlens, b),
                                   _varlen_heads(v, cu_seqlens, b), scale,
                                   causal=causal, window=window,
                                   dropout=_seq_dropout(dropout, b, H))
        o[lo:hi] = np.transpose(ob[0], (1, 0, 2))
        lse[:, lo:hi] = lb[0]
    return o, lse


def attention_backward_varlen(q, k, v, do, cu_seqlens, scale, causal=False,
                              window=None, dropout=None):
    """dQ, dK, dV [T,H,d], O [T,H,d] and LSE [H,T] of packed sequences, each
    sequence's gradient being that of its own attention."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    T, H, _ = q.shape
    dq, dk, dv, o = (np.zeros(x.shape) for x in (q, k, v, v))
    lse = np.full((H, T), -np.inf)
    for b in range(len(cu_seqlens) - 1):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if hi <= lo:
            continue
        r = attention_backward(*(_varlen_heads(x, cu_seqlens, b) for x in (q, k, v, do)),
                               scale, causal=causal, window=window,
                               dropout=_seq_dropout(dropout, b, H))
        for dst, src in zip((dq, dk, dv, o), r[:4]):
            dst[lo:hi] = np.transpose(src[0], (1, 0, 2))
        lse[:, lo:hi] = r[4][0]
    return dq, dk, dv, o, lse
