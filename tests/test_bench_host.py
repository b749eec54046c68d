"""Host-side checks of the benchmark's FLOP accounting (no GPU): forward
4*B*H*N^2*d, halved under the causal mask, scaled by the live-tile density
of a block mask; backward 2.5x the forward."""

import pytest

import bench
from exact_io_aware_tma_gb300.workloads import WORKLOADS


def band_global_live(T, band, every):
    # |i - j| <= band tiles (a band of width 2*band + 1, clipped at the
    # edges) plus every `every`-th key column, minus the band tiles that lie
    # in those columns: counted row by row
    live = 0
    for i in range(T):
        lo, hi = max(0, i - band), min(T - 1, i + band)
        in_band = hi - lo + 1
        glob = (T + every - 1) // every
        both = sum(1 for j in range(lo, hi + 1) if j % every == 0)
        live += in_band + glob - both
    return live


def test_band_global_count_of_the_block_sparse_workload():
    # 128 tile rows: 382 band tiles, 8 global columns of 128, 23 in both
    assert band_global_live(128, 1, 16) == 382 + 8 * 128 - 23 == 1383


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_flops_follow_the_formula(name):
    cfg = WORKLOADS[name]
    B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
    frac = {"causal": 0.5, "none": 1.0, "kv_len": 1.0}.get(cfg["mask"])
    if cfg["mask"] == "band_global":
        T = (N + 127) // 128
        frac = band_global_live(T, cfg["band"], cfg["global_every"]) / (T * T)
    want_fwd = 4.0 * B * H * N * N * d * frac
    fwd, bwd = bench.flops(cfg, bench.dense_fraction(cfg))
    assert fwd == pytest.approx(want_fwd, rel=1e-12)
    assert bwd == pytest.approx(2.5 * want_fwd, rel=1e-12)


def test_flops_of_the_five_workloads():
    # the forward counts of the tiny, BERT, GPT-2, long-context and
    # block-sparse shapes, to three significant digits
    want = {"tiny_dense_n128_d64": 4.19e6, "bert_large_keypad_n512_d64": 8.59e9,
            "gpt2_causal_n1024_d64": 1.29e10, "long_causal_n8192_d128": 5.50e11,
            "block_sparse_n16384_d64": 4.64e10}
    for name, w in want.items():
        cfg = WORKLOADS[name]
        fwd, _ = bench.flops(cfg, bench.dense_fraction(cfg))
        assert fwd == pytest.approx(w, rel=5e-3), name


def test_key_padding_effective_fraction():
    # BERT-shaped key padding: the effective pair fraction is the mean of
    # kv_len[b] / N, every drawn length within [256, 512]
    from exact_io_aware_tma_gb300.workloads import make_inputs
    cfg = WORKLOADS["bert_large_keypad_n512_d64"]
    inp = make_inputs(**cfg, with_grad=False)
    lens = [int(x) for x in inp["kv_len"]]
    assert all(256 <= x <= 512 for x in lens)
    want = sum(lens) / (len(lens) * cfg["N"])
    assert bench.effective_fraction(cfg, inp) == pytest.approx(want, rel=1e-15)
    assert 0.5 <= bench.effective_fraction(cfg, inp) <= 1.0
    # other masks report no effective figure
    for name in ("gpt2_causal_n1024_d64", "tiny_dense_n128_d64"):
        other = make_inputs(**WORKLOADS[name], with_grad=False)
        assert bench.effective_fraction(WORKLOADS[name], other) is None


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_both_arms_name_the_same_config(name):
    # the GPU arm and the oracle arm build `config` with one helper
    cfg = WORKLOADS[name]
    a = bench.workload_config(name, cfg, 1)
    assert a == bench.workload_config(name, dict(cfg), 1)
    assert a["workload"] == name and a["parallelism"] == "replicas1"
    assert {"B", "H", "N", "d", "mask", "l2"} <= set(a)


def test_datasheet_peak_matches_the_per_sm_rate():
    # 2.5 PFLOP/s dense (half the sparse per-GPU figure) is within 4% of
    # 152 SMs x 8192 dense bf16 FLOP per clock x the 2.07 GHz maximum clock
    derived = 152 * 8192 * 2.07e9 / 1e12
    assert bench.DATASHEET_BF16_TFLOPS == 2500.0
    assert abs(derived - bench.DATASHEET_BF16_TFLOPS) / derived < 0.04
