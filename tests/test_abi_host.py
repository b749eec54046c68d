"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol include/fa.h declares, and rejects bad arguments with status codes
before touching a GPU.  No compute call runs here."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_tma_gb300 import fa
    if not os.path.exists(fa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return fa.load()


def declared_symbols():
    out = []
    for h in HEADERS:
        out += re.findall(r"FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", open(h).read())
    return out


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    assert {"fa_forward", "fa_backward", "fa_backward_workspace_bytes",
            "fa_tile_schedule", "fa_status_string", "fa_last_device_status"} <= names


def test_library_exports_every_declared_symbol(lib):
    from exact_io_aware_tma_gb300 import fa
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in fa.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings(lib):
    from exact_io_aware_tma_gb300 import fa
    assert fa.status_string(0) == "FA_OK"
    assert fa.status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"


def test_workspace_is_linear_in_n(lib):
    # LSE*log2e and D (fp32 per row, rows padded to 128 per head) + fp32 dQ
    # accumulator, each rounded to 256 bytes, + 256 bytes for the dK/dV
    # kernel's work counter: no N x N term (the backward needs O(N) extra
    # memory per head).
    f = lib.fa_backward_workspace_bytes
    for B, H, N, d in [(1, 1, 128, 64), (2, 16, 8192, 128), (1, 8, 16384, 64), (3, 5, 7, 64)]:
        prow = B * H * (-(-N // 128) * 128)
        want = 2 * (-(-prow * 4 // 256) * 256) + -(-B * H * N * d * 4 // 256) * 256 + 256
        assert f(B, H, N, d) == want
    assert f(0, 1, 128, 64) == 0 and f(1, 1, 128, 96) == 0


FAKE = 1 << 20  # an aligned non-null address; never dereferenced on reject paths


def test_masked_workspace_adds_the_split_part_only_with_a_block_mask(lib):
    # plan items (16 B x 4 per key tile), 256 bytes of counts and split list,
    # 32 fp32 slots of 2 x 128 x d per head, each part rounded to 256 bytes;
    # nothing extra without a block mask or beyond 1024 key tiles
    from exact_io_aware_tma_gb300 import fa
    f = lib.fa_backward_workspace_bytes_masked
    for B, H, N, d in [(1, 8, 16384, 64), (2, 3, 300, 128), (1, 1, 1, 64)]:
        T = -(-N // 128)
        base = lib.fa_backward_workspace_bytes(B, H, N, d)
        extra = -(-T * 64 // 256) * 256 + 256 + B * H * 32 * 2 * 128 * d * 4
        bm = fa.Mask(0, -1, -1, ctypes.c_void_p(FAKE), None, 0.0, 0, 0)
        assert f(B, H, N, d, ctypes.byref(bm)) == base + extra
        plain = fa.Mask(1, -1, -1, None, None, 0.0, 0, 0)
        assert f(B, H, N, d, ctypes.byref(plain)) == base
        assert f(B, H, N, d, None) == base
    big = fa.Mask(0, -1, -1, ctypes.c_void_p(FAKE), None, 0.0, 0, 0)
    assert f(1, 1, 1025 * 128, 64, ctypes.byref(big)) == lib.fa_backward_workspace_bytes(
        1, 1, 1025 * 128, 64)
    assert f(1, 1, 128, 96, ctypes.byref(big)) == 0


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64,
         scale=0.125, causal=0, bm=None, kv=None):
    vp = ctypes.c_void_p
    return lib.fa_forward(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, N, d, scale,
                          causal, vp(bm) if bm else None, vp(kv) if kv else None, None)


def test_forward_rejects_bad_arguments(lib):
    assert _fwd(lib, d=96) == 2
    assert _fwd(lib, d=32) == 2
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, q=0) == 1
    assert _fwd(lib, lse=0) == 1
    assert _fwd(lib, k=FAKE + 8) == 1           # bf16 tensors need 16-byte alignment
    assert _fwd(lib, lse=FAKE + 2) == 1
    assert _fwd(lib, kv=FAKE + 1) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, scale=float("inf")) == 1
    assert _fwd(lib, B=65536, H=65536) == 1     # B*H beyond int32
    assert _fwd(lib, N=128 * 65536) == 1        # too many query tiles


def test_backward_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    ws = lib.fa_backward_workspace_bytes(1, 1, 128, 64)

    def bwd(ptrs=None, wsb=ws, d=64, wsp=FAKE):
        p = [FAKE] * 9 if ptrs is None else ptrs
        return lib.fa_backward(*[vp(x) for x in p], 1, 1, 128, d, 0.125, 0, None, None,
                               vp(wsp), wsb, None)

    assert bwd(d=80) == 2
    assert bwd(wsb=ws - 1) == 1
    assert bwd(wsp=0) == 1
    assert bwd(wsp=FAKE + 16) == 1              # workspace needs 256-byte alignment
    for i in range(9):
        p = [FAKE] * 9
        p[i] = 0
        assert bwd(p) == 1, i


def test_tile_schedule_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.fa_tile_schedule(0, 0, None, None, 0, vp(FAKE), vp(FAKE), vp(FAKE), None) == 1
    assert lib.fa_tile_schedule(256, 0, None, None, -1, vp(FAKE), vp(FAKE), vp(FAKE), None) == 1
    assert lib.fa_tile_schedule(256, 0, None, None, 0, None, vp(FAKE), vp(FAKE), None) == 1


def test_product_path_has_no_oracle_dependency():
    # The package and the CUDA sources never import, include or load the oracle.
    pkg = os.path.join(ROOT, "exact_io_aware_tma_gb300")
    pat = re.compile(r"^\s*(from\s+oracle|import\s+oracle|#include\s+.*oracle)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f


def test_binding_raises_without_library(tmp_path):
    from exact_io_aware_tma_gb300 import fa
    saved = fa._lib
    try:
        fa._lib = None
        with pytest.raises(RuntimeError):
            fa.load(str(tmp_path / "missing.so"))
    finally:
        fa._lib = saved
