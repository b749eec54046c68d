"""The forward's staged K/V ring: stage t carries V of the t-th live key tile
of a CTA's union and K of the next one on one full and one empty barrier,
and K of the first tile waits in the last stage's K slot ahead of that
stage's first use.  What the staging adds over a ring of single tiles is
checked here against the fp64 oracle: unions of one to five tiles (the
first K alone, a first stage without a next K, the last stage's first
reuse), two-tile CTAs whose union holds tiles live for only one of the two
query tiles (or for none of the pair at all), four stages at d = 64 (the
two-tile kernel of packed sequences longer than 2048), and the one-tile
d = 64 kernel with one, two and three live tiles per query tile.  Marked
``gpu``."""

import numpy as np
import pytest

from exact_io_aware_tma_gb300.workloads import make_inputs
from parity import compare_heads, run_gpu
from test_gpu_parity import oracle_on_heads
from test_gpu_varlen import run as run_varlen

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [128, 256, 384, 640])
@pytest.mark.parametrize("causal", [False, True])
def test_two_tile_unions_of_one_to_five_tiles(n, causal):
    # d = 128, two query tiles per CTA: the union has ceil(n / 128) tiles
    # (one to five), so the ring runs 0-4 stages past the first K
    inp = make_inputs(B=1, H=3, N=n, d=128, mask="causal" if causal else "none", seed=n + causal)
    heads = [(0, h) for h in range(3)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)


def test_two_tile_unions_with_one_sided_and_dead_tiles():
    # query tiles (rows) x key tiles (columns), pairs (0, 1) (2, 3) (4, 5)
    # (6, 7): tile 1 dead beside a one-tile tile 0; tiles live for one side
    # only, out of order; a dead pair; a full row beside a one-tile row
    T = 8
    bm = np.zeros((T, T), np.uint8)
    bm[0, 5] = 1
    bm[2, [0, 7]] = 1
    bm[3, 3] = 1
    bm[6, :] = 1
    bm[7, 6] = 1
    inp = make_inputs(B=1, H=2, N=T * 128, d=128, mask="none", seed=71)
    inp["block_mask"] = bm
    res = run_gpu(inp)
    heads = [(0, 0), (0, 1)]
    compare_heads(res, oracle_on_heads(inp, heads), heads)
    for qt in (1, 4, 5):
        rows = slice(qt * 128, (qt + 1) * 128)
        assert np.all(res["o"][:, :, rows] == 0) and np.all(np.isneginf(res["lse"][:, :, rows]))


@pytest.mark.parametrize("causal", [False, True])
def test_four_stages_at_d64(causal):
    # packed sequences longer than 2048 run the two-tile kernel at d = 64,
    # whose ring is four stages; 2432 rows = 19 key tiles, so each stage
    # barrier cycles several times, and 130 rows = a two-tile union
    run_varlen([2432, 700, 130], 2, 64, causal=causal, seed=72 + causal)


def test_one_tile_d64_with_one_two_and_three_live_tiles():
    # one-tile CTAs (d = 64, P apart): key lengths of one row, one tile, one
    # tile and a row, two tiles and a row
    inp = make_inputs(B=4, H=2, N=512, d=64, mask="none", seed=73)
    inp["kv_len"] = np.array([1, 128, 129, 257], np.int32)
    heads = [(b, h) for b in range(4) for h in range(2)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)


def test_one_tile_d64_block_mask_single_and_scattered_tiles():
    # one live key tile per query tile, then scattered live tiles with gaps
    # wider than a 32-tile bitmask word
    T = 40
    bm = np.zeros((T, T), np.uint8)
    for i in range(T):
        bm[i, (7 * i) % T] = 1
        if i % 3 == 0:
            bm[i, [0, min(T - 1, i + 33)]] = 1
    inp = make_inputs(B=1, H=1, N=T * 128, d=64, mask="none", seed=74)
    inp["block_mask"] = bm
    heads = [(0, 0)]
    compare_heads(run_gpu(inp), oracle_on_heads(inp, heads), heads)
