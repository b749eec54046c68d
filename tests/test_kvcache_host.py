"""Host-side checks of the key/value-cache entry points (include/fa_kvcache.h):
the split-count choice, the workspace size, and argument rejection before
any CUDA call.  No compute call runs here."""

import ctypes
import math

import pytest

FAKE = 1 << 20  # aligned non-null address; never dereferenced on reject paths
vp = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    import os
    from exact_io_aware_tma_gb300 import fa
    if not os.path.exists(fa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return fa.load()


@pytest.mark.parametrize("B,H,Nq,Nk,d", [(8, 16, 1, 32768, 128), (8, 16, 4, 32768, 128),
                                         (32, 12, 1, 4096, 64), (1, 1, 1, 64, 64),
                                         (1, 1, 3, 100000, 128), (64, 32, 1, 8192, 128),
                                         (2, 2, 9, 1000, 64)])
def test_split_choice_bounds(lib, B, H, Nq, Nk, d):
    S = lib.fa_kvcache_num_splits(B, H, Nq, Nk, d, 152)
    # at least one split, at most one per 256 keys and at most 256
    assert 1 <= S <= min(256, math.ceil(Nk / 256))
    # the choice is a pure function of its arguments
    assert S == lib.fa_kvcache_num_splits(B, H, Nq, Nk, d, 152)


def test_split_choice_items_per_resident_cta(lib):
    # one-row passes: 3 CTAs per SM, about 1.5 items per resident CTA
    # (456 on 152 SMs): 128 heads -> ceil(684 / 128) = 6, 384 heads -> 2
    assert lib.fa_kvcache_num_splits(8, 16, 1, 32768, 128, 152) == 6
    assert lib.fa_kvcache_num_splits(32, 12, 1, 4096, 64, 152) == 2
    # multi-row passes: 2 CTAs per SM, 8 items per resident CTA (304):
    # ceil(2432 / 128) = 19
    assert lib.fa_kvcache_num_splits(8, 16, 4, 32768, 128, 152) == 19
    # capped at one split per 256 keys
    assert lib.fa_kvcache_num_splits(1, 1, 1, 1000, 64, 152) == 4
    # Tiny caches are not split.
    assert lib.fa_kvcache_num_splits(1, 1, 1, 64, 64, 152) == 1
    assert lib.fa_kvcache_num_splits(1, 1, 1, 64, 96, 152) == 0


def test_workspace_bytes(lib):
    f = lib.fa_kvcache_workspace_bytes
    assert f(8, 16, 1, 32768, 128, 1) == 0
    for B, H, Nq, Nk, d, S in [(8, 16, 1, 32768, 128, 19), (2, 3, 5, 77, 64, 4),
                               (1, 1, 1, 1, 64, 256)]:
        rows = B * H * Nq
        want = (-(-S * rows * d * 4 // 256) * 256) + (-(-S * rows * 4 // 256) * 256)
        assert f(B, H, Nq, Nk, d, S) == want
    assert f(1, 1, 1, 64, 64, 257) == 0 and f(1, 1, 1, 64, 64, -1) == 0
    assert f(1, 1, 1, 64, 80, 2) == 0 and f(0, 1, 1, 64, 64, 2) == 0


def _kvc(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=1, Nk=128, d=64,
         scale=0.125, causal=0, cl=None, S=2, ws=FAKE, wsb=1 << 20):
    return lib.fa_forward_kvcache(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, Nq, Nk, d, scale,
                                  causal, vp(cl) if cl else None, S, vp(ws) if ws else None,
                                  wsb, None)


def test_forward_kvcache_rejects_bad_arguments(lib):
    assert _kvc(lib, d=96) == 2
    assert _kvc(lib, Nq=0) == 1 and _kvc(lib, Nk=0) == 1 and _kvc(lib, B=0) == 1
    assert _kvc(lib, q=0) == 1 and _kvc(lib, lse=0) == 1
    assert _kvc(lib, k=FAKE + 8) == 1          # bf16 tensors need 16-byte alignment
    assert _kvc(lib, lse=FAKE + 2) == 1
    assert _kvc(lib, cl=FAKE + 1) == 1
    assert _kvc(lib, scale=float("nan")) == 1
    assert _kvc(lib, S=-1) == 1 and _kvc(lib, S=257) == 1
    assert _kvc(lib, ws=0) == 1                # two splits need a workspace
    assert _kvc(lib, ws=FAKE + 16) == 1        # 256-byte aligned
    need = lib.fa_kvcache_workspace_bytes(1, 1, 1, 128, 64, 2)
    assert _kvc(lib, wsb=need - 1) == 1
    assert _kvc(lib, B=65536, H=65536) == 1


def test_combine_rejects_bad_arguments(lib):
    def comb(op=FAKE, lp=FAKE, S=2, rows=4, d=64, o=FAKE, lse=FAKE):
        return lib.fa_combine(vp(op), vp(lp), S, rows, d, vp(o), vp(lse), None)
    assert comb(S=0) == 1 and comb(rows=0) == 1
    assert comb(d=6) == 1 and comb(d=2048) == 1 and comb(d=0) == 1
    assert comb(op=0) == 1 and comb(o=0) == 1
    assert comb(op=FAKE + 4) == 1 and comb(o=FAKE + 2) == 1
