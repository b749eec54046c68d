"""GPU parity of packed variable-length sequences (forward and backward,
with causal and sliding-window masks) against the fp64 oracle through the
C ABI."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import to_f64
from oracle import attention_backward_varlen
from parity import TOL_GRAD, TOL_O, check_close, check_lse

pytestmark = pytest.mark.gpu


def packed_inputs(lens, H, d, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    total = int(sum(lens))
    x = [torch.randn((total, H, d), generator=g).to(torch.bfloat16) for _ in range(4)]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return x, cu


def run(lens, H, d, causal=False, window=None, seed=0):
    (q, k, v, do), cu = packed_inputs(lens, H, d, seed)
    dev = "cuda"
    gq, gk, gv, gdo = (t.to(dev) for t in (q, k, v, do))
    gcu = torch.from_numpy(cu).to(dev)
    mx = max(max(lens), 1)
    o, lse = fa.forward_varlen(gq, gk, gv, gcu, mx, causal=causal, window=window)
    dq, dk, dv = fa.backward_varlen(gq, gk, gv, o, lse, gdo, gcu, mx, causal=causal,
                                    window=window)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    scale = 1.0 / np.sqrt(d)
    ref = attention_backward_varlen(to_f64(q), to_f64(k), to_f64(v), to_f64(do), cu, scale,
                                    causal, window)
    got = [t.double().cpu().numpy() for t in (dq, dk, dv, o, lse)]
    for name, g_, r_, tol in (("dQ", got[0], ref[0], TOL_GRAD), ("dK", got[1], ref[1], TOL_GRAD),
                              ("dV", got[2], ref[2], TOL_GRAD), ("O", got[3], ref[3], TOL_O)):
        check_close(name, g_, r_, tol)
    check_lse(got[4], ref[4])


LENS = [[1], [130], [127, 128, 129], [300, 1, 513, 64], [5, 0, 700, 256, 2]]


@pytest.mark.parametrize("lens", LENS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(False, None), (True, None), (True, (100, 0)),
                                           (False, (64, 64))])
def test_packed_sequences(lens, d, causal, window):
    run(lens, 2, d, causal, window, seed=sum(lens) + d)


def test_packed_realistic_length_mix():
    # 16 sequences of 64..2048 tokens, causal, d = 128, 4 heads
    lens = list(np.random.default_rng(0).integers(64, 2049, size=16))
    run(lens, 4, 128, causal=True, seed=1)


def test_bad_offsets_are_reported_not_faulted():
    # decreasing offsets: clamped on the device, reported as FA_ERR_INVALID_ARG
    H, d = 2, 64
    (q, k, v, _), _ = packed_inputs([200], H, d, 3)
    cu = torch.tensor([0, 150, 90, 200], dtype=torch.int32, device="cuda")
    o, lse = fa.forward_varlen(q.cuda(), k.cuda(), v.cuda(), cu, 150)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_ERR_INVALID_ARG
    assert fa.last_device_status() == fa.FA_OK  # the word is cleared by the read


@pytest.mark.parametrize("lens", [[2048, 300], [2100, 1, 300]])
def test_packed_d64_on_both_sides_of_the_cta_shape_threshold(lens):
    # at d = 64 packed sequences run one query tile per CTA while the
    # longest is at most 2048 rows, a pair of query tiles per CTA beyond
    run(lens, 2, 64, causal=True, seed=len(lens))
