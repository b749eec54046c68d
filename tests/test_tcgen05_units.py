"""Unit checks of the tensor-core building blocks on one 128-row tile
(include/fa_selftest.h) against a float64 matmul of the same bf16 values.
Each mode is one operand path of the attention kernels."""

import pytest
import torch

from exact_io_aware_tma_gb300 import fa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,n", [(0, 128), (1, 64), (1, 128), (2, 64), (2, 128),
                                    (3, 64), (3, 128), (4, 64), (4, 128)])
def test_single_tile_mma(mode, n):
    g = torch.Generator().manual_seed(100 + 10 * mode + n)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(128, 128 if mode == 0 else n, generator=g).to(torch.bfloat16).cuda()
    c = fa.selftest_mma(mode, a, b, n)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    if mode == 0:
        ref = a.double() @ b.double().T
    elif mode == 4:
        ref = a.double().T @ b.double()
    else:
        ref = a.double() @ b.double()
    err = (c.double() - ref).abs().max().item()
    # fp32 accumulation of 128 exact bf16 products
    assert err <= 1e-5 * ref.abs().max().item() * 16, (mode, n, err)


def test_single_tile_mma_e4m3():
    # mode 5: both operands e4m3, c = a b^T; products of two e4m3 values are
    # exact in fp32, so only the fp32 accumulation order differs
    g = torch.Generator().manual_seed(555)
    a = (4 * torch.randn(128, 128, generator=g)).to(torch.float8_e4m3fn)
    b = (4 * torch.randn(128, 128, generator=g)).to(torch.float8_e4m3fn)
    c = fa.selftest_mma(5, a.view(torch.uint8).cuda(), b.view(torch.uint8).cuda(), 128)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    ref = a.to(torch.float64) @ b.to(torch.float64).T
    err = (c.double().cpu() - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() * 16, err


@pytest.mark.parametrize("mode,n", [(6, 64), (6, 128), (7, 64), (7, 128)])
def test_single_tile_mma_sw32_depth16(mode, n):
    # modes 6/7: one MMA of depth 16 over 32-byte-swizzled K-major operands
    # (a thread-written in mode 6, TMA-loaded in mode 7); c = a[:, :16] b[:, :16]^T
    g = torch.Generator().manual_seed(700 + 10 * mode + n)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(n, 128, generator=g).to(torch.bfloat16).cuda()
    c = fa.selftest_mma(mode, a, b, n)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    ref = a[:, :16].double() @ b[:, :16].double().T
    err = (c.double() - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() * 16, (mode, n, err)
