"""Pins for the FP8 oracle (oracle/fp8.py): e4m3 rounding against torch's
float8_e4m3fn conversion (a library routine) incl. subnormals and exact
ties, the grid's published facts, block scales and the quantisation error
bound, and attention on inputs that quantise exactly (then the FP8 reference
equals the exact one).  CPU only."""

import numpy as np
import pytest
import torch

from oracle import attention_forward
from oracle.fp8 import GRID, attention_forward_fp8, dequantize, quantize_blocks, round_e4m3


def torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_grid_facts():
    # 8-bit e4m3 (no infinities, one NaN code per sign): 127 non-negative
    # finite values, largest 448, smallest subnormal 2^-9, smallest normal 2^-6
    assert len(GRID) == 127 and GRID[-1] == 448.0
    assert GRID[1] == 2.0 ** -9 and GRID[8] == 2.0 ** -6
    assert np.all(np.diff(GRID) > 0)


@pytest.mark.parametrize("scale", [1e-4, 1e-2, 1.0, 30.0, 400.0])
def test_rounding_matches_torch(scale):
    x = (np.random.default_rng(int(scale * 1000)).standard_normal(20000) * scale)
    x = np.clip(x, -448, 448).astype(np.float32)
    assert np.array_equal(round_e4m3(x), torch_e4m3(x))


def test_ties_round_to_even():
    mids = ((GRID[:-1] + GRID[1:]) / 2).astype(np.float32)
    exact = mids.astype(np.float64) == (GRID[:-1] + GRID[1:]) / 2
    mids = mids[exact]
    got = round_e4m3(mids)
    assert np.array_equal(got, torch_e4m3(mids))
    assert np.array_equal(round_e4m3(-mids), -got)


def test_block_scale_and_error_bound():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((2, 3, 300, 64)) * 5).astype(np.float32)
    x[0, 0, 128:256] = 0.0  # an all-zero block
    codes, s = quantize_blocks(x, 128)
    assert s.shape == (2, 3, 3)
    assert s[0, 0, 1] == 1.0 and np.all(codes[0, 0, 128:256] == 0)
    # each block's largest element maps to +-448 exactly
    for t in range(3):
        blk = codes[1, 2, t * 128:(t + 1) * 128]
        assert np.abs(blk).max() == 448.0
    xr = dequantize(codes, s)
    ss = np.repeat(s, 128, axis=-1)[..., :300, None].astype(np.float64)
    bound = np.maximum(2.0 ** -4 * np.abs(x), ss * 2.0 ** -10)
    assert np.all(np.abs(xr - x) <= bound * (1 + 1e-6))


def test_blocks_are_independent():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((1, 1, 256, 64)).astype(np.float32)
    y = x.copy()
    y[0, 0, 200] *= 50  # only the second block changes
    cx, sx = quantize_blocks(x)
    cy, sy = quantize_blocks(y)
    assert np.array_equal(cx[0, 0, :128], cy[0, 0, :128]) and sx[0, 0, 0] == sy[0, 0, 0]
    assert sx[0, 0, 1] != sy[0, 0, 1]


def test_exactly_representable_inputs_give_exact_attention():
    # values that are e4m3 codes times the block scale 2^-3 (amax 448 * 2^-3
    # in every block) quantise without error: FP8 reference = exact reference
    rng = np.random.default_rng(3)
    B, H, N, d = 1, 2, 256, 64

    def exact_block_values():
        codes = rng.choice(np.concatenate([GRID, -GRID]), size=(B, H, N, d))
        codes[..., ::128, 0] = 448.0  # pin every block's amax at 448
        return (codes * 2.0 ** -3).astype(np.float32)

    q, k = exact_block_values(), exact_block_values()
    v = exact_block_values()
    o8, lse8, (qc, qs), _, _ = attention_forward_fp8(q, k, v, 0.01, causal=True)
    assert np.all(qs == 2.0 ** -3)
    o, lse = attention_forward(q, k, v, 0.01, causal=True)
    np.testing.assert_allclose(o8, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse8, lse, atol=1e-12, rtol=0)


def test_fp8_reference_is_close_to_exact():
    # Sanity scale of the quantisation itself: e4m3 keeps 3 mantissa bits, a
    # uniform relative rounding error of rms 2^-4/sqrt(3) ~ 3.6% per element,
    # so a score scale * q.k over d = 128 N(0,1) products moves by about
    # sqrt(2) * 3.6% ~ 0.05 (rms); over 600 rows the worst is a few times
    # that.  Bounds: LSE <= 0.25, O <= 10% of max |O|.
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((1, 2, 300, 128)).astype(np.float32) for _ in range(3))
    o8, lse8 = attention_forward_fp8(q, k, v, 128 ** -0.5, causal=True)[:2]
    o, lse = attention_forward(q, k, v, 128 ** -0.5, causal=True)
    assert np.abs(o8 - o).max() <= 0.10 * np.abs(o).max()
    assert np.abs(lse8 - lse).max() <= 0.25
