"""The backward's split of heavy key tiles (block masks): a key tile whose
column has many live query tiles is walked by several CTAs, whose partial
dK, dV rows land in the workspace's slots for a join kernel to add.  Checked against the oracle and
against the same call given only the unsplit workspace.  Marked ``gpu``."""

import numpy as np
import pytest
import torch

from exact_io_aware_tma_gb300 import fa
from exact_io_aware_tma_gb300.workloads import make_inputs
from oracle import dropout_p8
from parity import TOL_GRAD, check_close, compare_heads, to_device
from test_gpu_parity import oracle_on_heads

pytestmark = pytest.mark.gpu


def run_both(inp, dropout=None):
    """(split, unsplit) results of forward + backward on the same inputs."""
    g = to_device(inp)
    kw = dict(causal=g["causal"], block_mask=g["block_mask"], kv_len=g["kv_len"],
              scale=g["scale"], dropout=dropout)
    B, H, N, d = g["q"].shape
    o, lse = fa.forward(g["q"], g["k"], g["v"], **kw)
    full = fa.backward_workspace_bytes(B, H, N, d, g["block_mask"])
    base = fa.backward_workspace_bytes(B, H, N, d)
    assert full > base
    out = []
    for nbytes in (full, base):
        ws = torch.full((nbytes,), 0xAB, device="cuda", dtype=torch.uint8)
        dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], workspace=ws, **kw)
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        out.append({n: t.double().cpu().numpy()
                    for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()})
    return out


def agree(a, b):
    # the same sums in another order, each rounded to bf16 once
    for n in ("dq", "dk", "dv"):
        ref = np.abs(b[n]).max()
        assert np.abs(a[n] - b[n]).max() <= 1e-2 * ref, n


@pytest.mark.parametrize("d", [64, 128])
def test_global_columns_split_matches_unsplit_and_oracle(d):
    # 32 key tiles; every 8th is a global column (all 32 query tiles live),
    # so its work is four times the average and is split into parts
    inp = make_inputs(B=1, H=2, N=4096, d=d, mask="band_global", seed=31, global_every=8)
    split, unsplit = run_both(inp)
    agree(split, unsplit)
    compare_heads(split, oracle_on_heads(inp, [(0, 1)]), [(0, 1)])


def test_split_with_ragged_tail_dead_column_and_key_limit():
    # a ragged last tile, a key tile with no live query tile (its dK, dV are
    # 0), batch elements whose key limit cuts parts short or empties them
    n = 7 * 128 + 45
    inp = make_inputs(B=3, H=2, N=n, d=64, mask="none", seed=8)
    bm = np.zeros((8, 8), np.uint8)
    bm[:, 0] = 1
    bm[:, 5] = 1
    np.fill_diagonal(bm, 1)
    bm[3, 3] = 0
    bm[:, 3] = 0
    inp["block_mask"] = bm
    inp["kv_len"] = np.array([n, 700, 0], np.int32)
    split, unsplit = run_both(inp)
    agree(split, unsplit)
    heads = [(b, h) for b in range(3) for h in range(2)]
    compare_heads(split, oracle_on_heads(inp, heads), heads)
    assert np.all(split["dk"][:, :, 384:512] == 0) and np.all(split["dv"][:, :, 384:512] == 0)
    assert np.all(split["dk"][2] == 0) and np.all(split["dv"][2] == 0)


def test_split_with_dropout():
    inp = make_inputs(B=1, H=2, N=1024, d=64, mask="band_global", seed=12, global_every=4)
    drop = dict(p=0.2, seed=777, offset=3)
    split, unsplit = run_both(inp, dropout=(drop["p"], drop["seed"], drop["offset"]))
    agree(split, unsplit)
    inp["dropout"] = drop
    heads = [(0, 0), (0, 1)]
    compare_heads(split, oracle_on_heads(inp, heads), heads)
    assert dropout_p8(drop["p"]) == 51


def test_split_repeats_bit_exactly():
    # the join adds the slots in part order, so a repeated call gives the
    # same bits whatever order the parts ran in
    inp = make_inputs(B=1, H=4, N=2048, d=128, mask="band_global", seed=2, global_every=4)
    a, _ = run_both(inp)
    b, _ = run_both(inp)
    for n in ("dq", "dk", "dv"):
        if n == "dq":
            # dQ is accumulated with atomics across CTAs: order-dependent
            check_close(n, a[n], b[n], TOL_GRAD)
        else:
            assert np.array_equal(a[n], b[n]), n


def test_three_launch_entry_points_split_like_the_one_call():
    # fa_backward_preprocess / fa_backward_dkdv / fa_backward_dq_convert with
    # the masked workspace (the dK/dV entry plans and splits by itself) give
    # the one-call backward's results bit for bit in dK, dV
    inp = make_inputs(B=1, H=3, N=2048, d=64, mask="band_global", seed=21, global_every=4)
    g = to_device(inp)
    B, H, N, d = g["q"].shape
    o, lse = fa.forward(g["q"], g["k"], g["v"], block_mask=g["block_mask"], scale=g["scale"])
    dq1, dk1, dv1 = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"],
                                block_mask=g["block_mask"], scale=g["scale"])
    lib, P = fa.load(), fa._ptr
    wsb = fa.backward_workspace_bytes(B, H, N, d, g["block_mask"])
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    dq2, dk2, dv2 = (torch.empty_like(g["q"]) for _ in range(3))
    sp = fa._stream()
    assert lib.fa_backward_preprocess(P(o), P(g["do"]), P(lse), B, H, N, d, P(ws), wsb, sp) == 0
    assert lib.fa_backward_dkdv(P(g["q"]), P(g["k"]), P(g["v"]), P(g["do"]), P(dk2), P(dv2), B, H,
                                N, d, g["scale"], 0, P(g["block_mask"]), None, P(ws), wsb,
                                sp) == 0
    assert lib.fa_backward_dq_convert(P(dq2), B, H, N, d, g["scale"], P(ws), wsb, sp) == 0
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    check_close("dQ", dq2.double().cpu().numpy(), dq1.double().cpu().numpy(), TOL_GRAD)
