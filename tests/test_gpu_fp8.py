"""GPU checks of the FP8 forward with block quantisation (include/fa_fp8.h)
against the fp64 oracle (oracle/fp8.py): the e4m3 codes and block scales bit
for bit, then O and LSE of the attention kernel against exact attention on
the dequantised operands, with a bound derived from the kernel's one extra
rounding (its probabilities are rounded to e4m3 for the P V product)."""

import math

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs, to_f64
from oracle import allowed_mask, attention_forward
from oracle.fp8 import attention_forward_fp8, dequantize, quantize_blocks

pytestmark = pytest.mark.gpu


def e4m3_values(u8):
    return u8.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("N", [128, 300, 1000])
def test_quantisation_bit_exact(N):
    inp = make_inputs(B=2, H=2, N=N, d=128, mask="none", seed=N)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    ws = fa.fp8_quantize(q, k, v)
    torch.cuda.synchronize()
    views = fa.fp8_workspace_views(ws, 2, 2, N)
    _, _, (qc, qs), (kc, ks), (vc, vs) = attention_forward_fp8(
        inp["q"].float().numpy(), inp["k"].float().numpy(), inp["v"].float().numpy(), 0.1)
    T = (N + 127) // 128
    assert np.array_equal(e4m3_values(views["q8"]).reshape(2, 2, N, 128), qc)
    assert np.array_equal(e4m3_values(views["k8"]).reshape(2, 2, N, 128), kc)
    vt = e4m3_values(views["vt8"]).reshape(2, 2, 128, T * 128)
    assert np.array_equal(np.swapaxes(vt[..., :N], -1, -2), vc)
    assert np.all(vt[..., N:] == 0)
    assert np.array_equal(views["qs"].cpu().numpy().reshape(2, 2, T), qs)
    assert np.array_equal(views["ks"].cpu().numpy().reshape(2, 2, T), ks)
    assert np.array_equal(views["vs"].cpu().numpy().reshape(2, 2), vs[..., 0])


def test_quantisation_bit_exact_every_scale_significand():
    # The division by the block scale in the quantisation kernels: one head
    # per bf16 significand of amax (128) at amax exponents -125 (scale below
    # the fp32 normal range), -100, 0 and 100, each head holding amax and
    # every bf16 value from amax * 2^-24 up to amax (both signs): every
    # quotient's e4m3 code and every scale must equal the oracle's fp32
    # division.
    rng = np.random.default_rng(5)
    heads = []
    for e in (-125, -100, 0, 100):
        for m in range(128):
            amax = (1 + m / 128) * 2.0 ** e
            vals = np.array([(1 + mm / 128) * 2.0 ** ee for ee in range(e - 24, e + 1)
                             for mm in range(128)])
            vals = vals[(vals <= amax) & (vals >= 2.0 ** -126)]
            vals = np.concatenate([vals, -vals])
            blk = np.resize(rng.permutation(vals), 128 * 128)
            blk[rng.integers(128 * 128)] = amax
            heads.append(blk.reshape(128, 128))
    x = torch.from_numpy(np.stack(heads)[None]).to(torch.bfloat16)
    H = x.shape[1]
    assert np.array_equal(x.double().numpy(), np.stack(heads)[None])  # values are bf16
    xd = x.cuda()
    ws = fa.fp8_quantize(xd, xd, xd)
    torch.cuda.synchronize()
    views = fa.fp8_workspace_views(ws, 1, H, 128)
    codes, scales = quantize_blocks(x.float().numpy())
    for name, sname in (("q8", "qs"), ("k8", "ks")):
        assert np.array_equal(e4m3_values(views[name]).reshape(1, H, 128, 128), codes), name
        assert np.array_equal(views[sname].cpu().numpy().reshape(1, H, 1), scales), sname
    vt = e4m3_values(views["vt8"]).reshape(1, H, 128, 128)
    assert np.array_equal(np.swapaxes(vt, -1, -2), codes)
    assert np.array_equal(views["vs"].cpu().numpy().reshape(1, H), scales[..., 0])


@pytest.mark.parametrize("N,causal", [(128, False), (300, True), (1000, True), (1000, False),
                                      (2048, True)])
def test_fp8_forward_parity(N, causal):
    B, H, d = 1, 2, 128
    inp = make_inputs(B=B, H=H, N=N, d=d, mask="none", seed=N + 7)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward_fp8(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    qf, kf, vf = (inp[x].float().numpy() for x in ("q", "k", "v"))
    ro, rlse, (qc, qs), (kc, ks), (vc, vs) = attention_forward_fp8(qf, kf, vf, scale, causal)
    # LSE: scores are exact products of e4m3 codes summed in fp32
    assert np.abs(lse - rlse).max() <= 1e-3
    # O: the kernel rounds each probability to e4m3 (relative error uniform
    # within +-2^-4, rms 2^-4/sqrt(3)) in the P V product while l keeps the
    # unrounded sum.  Per row, the error of O is then about that rms times
    # ||P_i||_2 * |V| from the numerator, plus as much from the mismatch of
    # the normaliser; the bound takes 8 sigma of both together over max|V^|,
    # plus the bf16 output rounding.
    qh, kh, vh = dequantize(qc, qs), dequantize(kc, ks), dequantize(vc, vs, None)
    rms = 2.0 ** -4 / math.sqrt(3)
    for h in range(H):
        s = scale * qh[0, h] @ kh[0, h].T
        ok = allowed_mask(N, None, causal)
        s = np.where(ok, s, -np.inf)
        pr = np.exp(s - s.max(1, keepdims=True))
        pr /= pr.sum(1, keepdims=True)
        pnorm = np.sqrt((pr ** 2).sum(1))
        bound = 8 * rms * math.sqrt(2) * pnorm * np.abs(vh[0, h]).max() + \
            2.0 ** -8 * np.abs(ro[0, h]).max(1) + 1e-4
        err = np.abs(o[0, h] - ro[0, h]).max(1)
        assert np.all(err <= bound), (h, float((err / bound).max()))
    # and the whole FP8 path against exact attention on the bf16 inputs
    eo, _ = attention_forward(to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]), scale,
                              causal=causal)
    assert np.abs(o - eo).max() <= 0.15 * np.abs(eo).max()


def test_fp8_rejects_unsupported_head_dim():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(q, q, q)
    assert e.value.status in (fa.FA_ERR_UNSUPPORTED, fa.FA_ERR_INVALID_ARG)
