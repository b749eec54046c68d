"""fp64 reference for the FP8 forward with block quantisation -- TEST
INFRASTRUCTURE ONLY (imported by tests, the smoke check and the benchmark's
CPU leg; never by the product path).

What the pages say (page "FlashAttention" (aiwiki), section "Development
across generations"): the Hopper generation's FP8 path adds block
quantisation and processing to reduce quantisation error, and such
low-precision execution is to be told apart from exact attention at higher
precision.  They give no formula.  Reading taken here (the plainest one):

* e4m3: the 8-bit float with 1 sign, 4 exponent (bias 7) and 3 mantissa
  bits, largest finite value 448, subnormals down to 2^-9.
* Q and K are quantised per block of 128 rows of one (b, h): the block's
  scale is s = amax / 448 (amax = the largest |x| of the block, both in
  fp32; s = 1 for an all-zero block) and each element's code is x / s (fp32
  division) rounded to the nearest e4m3 value, ties to even.  V is
  quantised the same way with one block per (b, h) (the whole head), so its
  scale factors out of the P V product.
* Attention is then the exact definition on the dequantised operands
  code * s:  O = softmax(scale * Q^ K^T) V^,  LSE as usual.  (The GPU path
  also rounds P to e4m3 before its P V product; that error is not part of
  the reference, it is what the FP8 tolerance covers.)
"""

import numpy as np

from .attention import attention_forward

E4M3_MAX = 448.0


def _e4m3_grid():
    """All non-negative finite e4m3 values, ascending (exact in fp64)."""
    vals = [m / 8.0 * 2.0 ** -6 for m in range(8)]            # subnormals
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                                       # NaN code
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


GRID = _e4m3_grid()


def round_e4m3(x):
    """Round fp32/fp64 values to the nearest e4m3 value, ties to the even
    mantissa, saturating at +-448 (inputs here never exceed it by more than
    rounding)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(GRID, a, side="left")
    hi = np.minimum(hi, len(GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    vlo, vhi = GRID[lo], GRID[hi]
    take_hi = (vhi - a) < (a - vlo)
    tie = (vhi - a) == (a - vlo)
    # even mantissa = even index in the grid (codes are consecutive)
    take_hi = take_hi | (tie & (hi % 2 == 0))
    r = np.where(a == vhi, vhi, np.where(take_hi, vhi, vlo))
    return np.sign(x) * r


def quantize_blocks(x, block=128):
    """x [..., N, d] (values as the GPU sees them) -> (codes as float64 e4m3
    values, scales [..., ceil(N / block)] fp32).  block=None: one block over
    the whole [N, d] matrix."""
    x = np.asarray(x, dtype=np.float32)
    N = x.shape[-2]
    blk = N if block is None else block
    nb = (N + blk - 1) // blk
    codes = np.zeros(x.shape, dtype=np.float64)
    scales = np.zeros(x.shape[:-2] + (nb,), dtype=np.float32)
    for t in range(nb):
        sl = x[..., t * blk:(t + 1) * blk, :]
        amax = np.abs(sl).max(axis=(-2, -1)).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[..., t] = s
        q = (sl / s[..., None, None]).astype(np.float32)
        codes[..., t * blk:(t + 1) * blk, :] = round_e4m3(q)
    return codes, scales


def dequantize(codes, scales, block=128):
    N = codes.shape[-2]
    blk = N if block is None else block
    s = np.repeat(scales.astype(np.float64), blk, axis=-1)[..., :N]
    return codes * s[..., None]


def attention_forward_fp8(q, k, v, scale, causal=False):
    """O, LSE of exact attention on the block-quantised operands (Q, K per
    128-row block, V per head).  Returns (o, lse, (qc, qs), (kc, ks), (vc, vs))."""
    qc, qs = quantize_blocks(q, 128)
    kc, ks = quantize_blocks(k, 128)
    vc, vs = quantize_blocks(v, None)
    o, lse = attention_forward(dequantize(qc, qs), dequantize(kc, ks),
                               dequantize(vc, vs, None), scale, causal=causal)
    return o, lse, (qc, qs), (kc, ks), (vc, vs)
