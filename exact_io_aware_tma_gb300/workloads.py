"""Seeded synthetic attention workloads.

This module draws inputs only; it holds none of the attention arithmetic, so
both the CUDA path and the fp64 oracle can be fed from it.

Recipe (same for every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``; draw Q, K, V, dO in that
    order, each iid N(0, 1) in fp32 of shape [B, H, N, d], then round to bf16
    (round-to-nearest-even, ``Tensor.to``).  Both sides see these bf16 values.
  * key padding: per batch row a valid key count drawn with
    ``numpy.random.default_rng(seed).integers(lo, hi + 1, size=B)``.
  * block mask over 128x128 tiles: a diagonal band |i - j| <= 1 (in tiles)
    united with global key columns j % 16 == 0.
  * scale = 1 / sqrt(d).
"""

import math

import numpy as np
import torch

TILE = 128

# name -> shape and mask structure.  The first is the small case the fp64
# oracle finishes in well under a second; the fourth is the long-context
# d=128 causal case the throughput is quoted on.
WORKLOADS = {
    "tiny_dense_n128_d64": dict(B=1, H=1, N=128, d=64, mask="none", seed=0),
    "bert_large_keypad_n512_d64": dict(B=8, H=16, N=512, d=64, mask="kv_len",
                                       kv_lo=256, kv_hi=512, seed=1),
    "gpt2_causal_n1024_d64": dict(B=8, H=12, N=1024, d=64, mask="causal",
                                  seed=2),
    "long_causal_n8192_d128": dict(B=2, H=16, N=8192, d=128, mask="causal",
                                   seed=3),
    "block_sparse_n16384_d64": dict(B=1, H=8, N=16384, d=64,
                                    mask="band_global", band=1, global_every=16,
                                    seed=4),
}

BENCH_WORKLOAD = "long_causal_n8192_d128"

# Attention of new query rows against a key/value cache: name -> shape.  The
# valid cache length of each batch row is drawn in [len_lo, len_hi]; slots
# past it hold random values that must not reach the result.
KVCACHE_WORKLOADS = {
    "decode_kvcache_b8_h16_nk32768_d128": dict(B=8, H=16, Nq=1, Nk=32768, d=128,
                                               causal=False, len_lo=16384,
                                               len_hi=32768, seed=5),
    "specdecode_kvcache_b8_h16_nq4_nk32768_d128": dict(B=8, H=16, Nq=4, Nk=32768,
                                                       d=128, causal=True,
                                                       len_lo=16384, len_hi=32768,
                                                       seed=6),
    "decode_kvcache_b32_h12_nk4096_d64": dict(B=32, H=12, Nq=1, Nk=4096, d=64,
                                              causal=False, len_lo=1024,
                                              len_hi=4096, seed=7),
}

KVCACHE_BENCH_WORKLOAD = "decode_kvcache_b8_h16_nk32768_d128"

# Masks beyond the five workloads above: a causal sliding window of 1024 keys
# on the long-context shape, a packed batch of 16 causal sequences whose
# lengths are drawn in [512, 8192] (numpy default_rng(seed)), dropout
# (p = 0.1, generator seed 2024) on the long-context shape, and the FP8
# forward on the long-context shape.
MASK_WORKLOADS = {
    "sliding_window_causal_n8192_d128_w1024": dict(B=2, H=16, N=8192, d=128, mask="causal",
                                                   window=(1023, 0), seed=8),
    "varlen_packed_causal_16seq_d128": dict(nseq=16, H=16, d=128, len_lo=512, len_hi=8192,
                                            causal=True, seed=9),
    "dropout_causal_n8192_d128_p0.1": dict(B=2, H=16, N=8192, d=128, mask="causal",
                                           dropout=(0.1, 2024, 0), seed=10),
    "fp8_forward_causal_n8192_d128": dict(B=2, H=16, N=8192, d=128, mask="causal", fp8=True,
                                          seed=11),
}


def band_global_block_mask(n_tiles, band=1, global_every=16):
    """uint8 [T, T]: 1 where |i - j| <= band or j % global_every == 0."""
    i = np.arange(n_tiles)[:, None]
    j = np.arange(n_tiles)[None, :]
    return ((np.abs(i - j) <= band) | (j % global_every == 0)).astype(np.uint8)


def make_inputs(B, H, N, d, mask="none", seed=0, kv_lo=None, kv_hi=None,
                band=1, global_every=16, with_grad=True):
    """Return a dict of CPU tensors / arrays for one workload.

    keys: q, k, v, do (bf16 [B,H,N,d]; do only if ``with_grad``), causal
    (bool), block_mask (uint8 numpy [T,T] or None), kv_len (int32 numpy [B]
    or None), scale (float).
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = (torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
          if with_grad else None)
    causal = mask == "causal"
    block_mask = None
    kv_len = None
    if mask == "band_global":
        t = (N + TILE - 1) // TILE
        block_mask = band_global_block_mask(t, band, global_every)
    elif mask == "kv_len":
        rng = np.random.default_rng(seed)
        kv_len = rng.integers(kv_lo, kv_hi + 1, size=B).astype(np.int32)
    elif mask not in ("none", "causal"):
        raise ValueError(f"unknown mask kind {mask!r}")
    return dict(q=q, k=k, v=v, do=do, causal=causal, block_mask=block_mask,
                kv_len=kv_len, scale=1.0 / math.sqrt(d))


def make_kvcache_inputs(B, H, Nq, Nk, d, causal=False, seed=0, len_lo=None,
                        len_hi=None):
    """CPU inputs for attention against a cache.

    ``torch.Generator('cpu').manual_seed(seed)``; Q [B,H,Nq,d], then K and V
    [B,H,Nk,d], iid N(0, 1) in fp32 rounded to bf16; cache_len (int32 [B])
    from ``numpy.random.default_rng(seed).integers(len_lo, len_hi + 1)``, or
    None (every slot valid) when ``len_lo`` is None.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    cache_len = None
    if len_lo is not None:
        rng = np.random.default_rng(seed)
        cache_len = rng.integers(len_lo, len_hi + 1, size=B).astype(np.int32)
    return dict(q=q, k=k, v=v, causal=bool(causal), cache_len=cache_len,
                scale=1.0 / math.sqrt(d))


def make_varlen_inputs(nseq, H, d, len_lo, len_hi, causal=True, seed=0):
    """Packed inputs: sequence lengths from ``numpy.random.default_rng(seed)
    .integers(len_lo, len_hi + 1, nseq)``, then Q, K, V, dO [total, H, d] iid
    N(0, 1) fp32 -> bf16 from ``torch.Generator('cpu').manual_seed(seed)``."""
    lens = np.random.default_rng(seed).integers(len_lo, len_hi + 1, size=nseq)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = [torch.randn((total, H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
         for _ in range(4)]
    return dict(q=x[0], k=x[1], v=x[2], do=x[3], cu_seqlens=cu, max_seqlen=int(lens.max()),
                causal=bool(causal), scale=1.0 / math.sqrt(d))


def kvcache_workload_inputs(name):
    return make_kvcache_inputs(**KVCACHE_WORKLOADS[name])


def workload_inputs(name, with_grad=True):
    return make_inputs(**WORKLOADS[name], with_grad=with_grad)


def to_f64(t):
    """bf16 torch tensor -> fp64 numpy copy (exact: bf16 embeds in fp64)."""
    return t.to(torch.float64).numpy()
