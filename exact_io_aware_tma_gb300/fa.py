"""ctypes binding of ``libfa_gb300.so`` (C ABI declared in include/fa.h,
include/fa_kvcache.h and include/fa_fp8.h).

Argument marshalling only: every step of attention runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  If the
library is missing, every call raises -- there is no fallback path.
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)

_lib = None

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_status_string": ([_i], ctypes.c_char_p),
    "fa_forward": ([_vp] * 5 + [_i] * 4 + [_f, _i, _vp, _vp, _vp], _i),
    "fa_backward_workspace_bytes": ([_i] * 4, _sz),
    "fa_backward_workspace_bytes_masked": ([_i] * 4 + [_vp], _sz),
    "fa_backward": ([_vp] * 9 + [_i] * 4 + [_f, _i, _vp, _vp, _vp, _sz, _vp], _i),
    "fa_backward_preprocess": ([_vp, _vp, _vp] + [_i] * 4 + [_vp, _sz, _vp], _i),
    "fa_backward_dkdv": ([_vp] * 6 + [_i] * 4 + [_f, _i, _vp, _vp, _vp, _sz, _vp], _i),
    "fa_backward_dq_convert": ([_vp] + [_i] * 4 + [_f, _vp, _sz, _vp], _i),
    "fa_tile_schedule": ([_i, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp], _i),
    "fa_last_device_status": ([_vp], _i),
    "fa_selftest_mma": ([_i, _vp, _vp, _vp, _i, _vp], _i),
    "fa_selftest_forward_lost_signal": ([_vp] * 5 + [_i] * 4 + [_f, _i, _vp], _i),
    "fa_selftest_backward_lost_signal": ([_vp] * 9 + [_i] * 4 + [_f, _i, _vp, _sz, _vp], _i),
    "fa_backward_noalloc": ([_vp] * 9 + [_i] * 4 + [_f, _i, _vp, _vp, _vp], _i),
    "fa_forward_masked": ([_vp] * 5 + [_i] * 4 + [_f, _vp, _vp], _i),
    "fa_backward_masked": ([_vp] * 9 + [_i] * 4 + [_f, _vp, _vp, _sz, _vp], _i),
    "fa_tile_schedule_masked": ([_i, _vp, _i, _vp, _vp, _vp, _vp], _i),
    "fa_forward_varlen": ([_vp] * 6 + [_i] * 5 + [_f, _vp, _vp], _i),
    "fa_varlen_workspace_bytes": ([_i] * 5, _sz),
    "fa_backward_varlen": ([_vp] * 10 + [_i] * 5 + [_f, _vp, _vp, _sz, _vp], _i),
    "fa_fp8_workspace_bytes": ([_i] * 4, _sz),
    "fa_fp8_quantize": ([_vp] * 3 + [_i] * 4 + [_vp, _sz, _vp], _i),
    "fa_forward_fp8_quantized": ([_vp, _vp, _vp] + [_i] * 4 + [_f, _i, _vp], _i),
    "fa_forward_fp8": ([_vp] * 5 + [_i] * 4 + [_f, _i, _vp, _sz, _vp], _i),
    "fa_kvcache_num_splits": ([_i] * 6, _i),
    "fa_kvcache_workspace_bytes": ([_i] * 6, _sz),
    "fa_forward_kvcache": ([_vp] * 5 + [_i] * 5 + [_f, _i, _vp, _i, _vp, _sz, _vp], _i),
    "fa_combine": ([_vp, _vp, _i, ctypes.c_longlong, _i, _vp, _vp, _vp], _i),
}

KVCACHE_MAX_SPLITS = 256  # FA_KVCACHE_MAX_SPLITS (include/fa_kvcache.h)

# Size of the library's built-in backward scratch (include/fa.h).
NOALLOC_SCRATCH_BYTES = 32 << 20


class Mask(ctypes.Structure):
    """``fa_mask`` of include/fa.h: every mask option of the *_masked calls
    (including dropout and its generator state)."""
    _fields_ = [("causal", ctypes.c_int), ("window_left", ctypes.c_int),
                ("window_right", ctypes.c_int), ("block_mask", ctypes.c_void_p),
                ("kv_len", ctypes.c_void_p), ("dropout_p", ctypes.c_float),
                ("dropout_seed", ctypes.c_uint64), ("dropout_offset", ctypes.c_uint32)]


class FAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load(path=LIB_PATH):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA attention library not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(status):
    return load().fa_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_qkv(*ts):
    ref = ts[0]
    for t in ts:
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("tensors must be contiguous bf16 CUDA tensors")
        if t.shape != ref.shape or t.dim() != 4:
            raise ValueError("tensors must share one [B, H, N, d] shape")


def _mask_args(N, block_mask, kv_len, B):
    T = (N + 127) // 128
    if block_mask is not None:
        if not (block_mask.is_cuda and block_mask.dtype == torch.uint8
                and block_mask.is_contiguous() and tuple(block_mask.shape) == (T, T)):
            raise ValueError(f"block_mask must be a contiguous uint8 CUDA [{T},{T}] tensor")
    if kv_len is not None:
        if not (kv_len.is_cuda and kv_len.dtype == torch.int32
                and kv_len.is_contiguous() and tuple(kv_len.shape) == (B,)):
            raise ValueError(f"kv_len must be a contiguous int32 CUDA [{B}] tensor")
    return _ptr(block_mask), _ptr(kv_len)


def _mask(N, causal, block_mask, kv_len, B, window, dropout=None):
    """``dropout`` = (p, seed, offset) or None."""
    bm, kl = _mask_args(N, block_mask, kv_len, B)
    wl, wr = (-1, -1) if window is None else (
        -1 if window[0] is None else int(window[0]), -1 if window[1] is None else int(window[1]))
    dp, seed, off = (0.0, 0, 0) if dropout is None else dropout
    return Mask(int(bool(causal)), wl, wr, bm, kl, float(dp), int(seed) & (2**64 - 1),
                int(off) & 0xFFFFFFFF)


def forward(q, k, v, causal=False, block_mask=None, kv_len=None, scale=None,
            out=None, lse=None, stream=None, window=None, dropout=None):
    """O, LSE = attention(q, k, v); see include/fa.h ``fa_forward_masked``.
    ``window`` = (left, right): key j allowed for query i only if
    i - left <= j <= i + right (None or negative = unbounded side).
    ``dropout`` = (p, seed, offset): dropout on P with the mask regenerated
    from (seed, offset) -- pass the same triple to ``backward``."""
    lib = load()
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32) if lse is None else lse
    m = _mask(N, causal, block_mask, kv_len, B, window, dropout)
    st = lib.fa_forward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                               scale, ctypes.byref(m), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_forward_masked")
    return out, lse


def backward_workspace_bytes(B, H, N, d, block_mask=None):
    """Workspace of a backward call; with a block mask, the larger size that
    lets the backward split heavy key tiles (``fa_backward_workspace_bytes_masked``)."""
    if block_mask is None:
        return int(load().fa_backward_workspace_bytes(B, H, N, d))
    m = _mask(N, False, block_mask, None, B, None)
    return int(load().fa_backward_workspace_bytes_masked(B, H, N, d, ctypes.byref(m)))


def backward(q, k, v, o, lse, do, causal=False, block_mask=None, kv_len=None,
             scale=None, workspace=None, dq=None, dk=None, dv=None, stream=None, window=None,
             dropout=None):
    """dQ, dK, dV of sum(O * dO); see include/fa.h ``fa_backward_masked``."""
    lib = load()
    _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = backward_workspace_bytes(B, H, N, d, block_mask)
    if workspace is None:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    m = _mask(N, causal, block_mask, kv_len, B, window, dropout)
    st = lib.fa_backward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, scale,
                                ctypes.byref(m), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_backward_masked")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    """Autograd node over ``forward`` / ``backward``: saves Q, K, V, O and the
    LSE (no P: the backward rebuilds it), nothing else."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale, block_mask, kv_len, window, dropout):
        o, lse = forward(q, k, v, causal=causal, block_mask=block_mask, kv_len=kv_len,
                         scale=scale, window=window, dropout=dropout)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.args = (causal, scale, block_mask, kv_len, window, dropout)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        causal, scale, block_mask, kv_len, window, dropout = ctx.args
        dq, dk, dv = backward(q, k, v, o, lse, do.contiguous(), causal=causal,
                              block_mask=block_mask, kv_len=kv_len, scale=scale, window=window,
                              dropout=dropout)
        return dq, dk, dv, None, None, None, None, None, None


def attention(q, k, v, causal=False, scale=None, block_mask=None, kv_len=None, window=None,
              dropout=None, return_lse=False):
    """Differentiable exact attention: O = softmax(scale * Q K^T [masked]) V
    for bf16 CUDA tensors [B, H, N, d], with the gradient of Q, K and V
    computed by ``backward`` when autograd asks for it.  Arguments as in
    ``forward``; returns O, or (O, LSE) with ``return_lse``."""
    o, lse = _Attention.apply(q, k, v, causal, scale, block_mask, kv_len, window, dropout)
    return (o, lse) if return_lse else o


def backward_noalloc(q, k, v, o, lse, do, causal=False, block_mask=None, kv_len=None,
                     scale=None, dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV like ``backward`` but with no workspace: the library's
    built-in scratch is used (``fa_backward_noalloc``; problems needing more
    than NOALLOC_SCRATCH_BYTES of workspace are rejected).  Output tensors
    are allocated here unless given; pass ``dq``/``dk``/``dv`` to allocate
    nothing at all."""
    lib = load()
    _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    bm, kl = _mask_args(N, block_mask, kv_len, B)
    st = lib.fa_backward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, scale,
                                 int(bool(causal)), bm, kl, _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_backward_noalloc")
    return dq, dk, dv


def _check_packed(*ts):
    ref = ts[0]
    for t in ts:
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 3):
            raise ValueError("packed tensors must be contiguous [total, H, d] bf16 CUDA tensors")
        if t.shape != ref.shape:
            raise ValueError("packed tensors must share one [total, H, d] shape")


def _check_cu(cu_seqlens):
    if not (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32
            and cu_seqlens.is_contiguous() and cu_seqlens.dim() == 1 and cu_seqlens.numel() >= 2):
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA [B+1] tensor")
    return cu_seqlens.numel() - 1


def forward_varlen(q, k, v, cu_seqlens, max_seqlen, causal=False, window=None, scale=None,
                   out=None, lse=None, stream=None, dropout=None):
    """O [total,H,d], LSE [H,total] of packed sequences; see ``fa_forward_varlen``."""
    lib = load()
    _check_packed(q, k, v)
    B = _check_cu(cu_seqlens)
    total, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), device=q.device, dtype=torch.float32) if lse is None else lse
    m = _mask(1, causal, None, None, 0, window, dropout)
    st = lib.fa_forward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
                               B, H, total, int(max_seqlen), d, scale, ctypes.byref(m),
                               _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_forward_varlen")
    return out, lse


def varlen_workspace_bytes(B, H, total, max_seqlen, d):
    return int(load().fa_varlen_workspace_bytes(B, H, total, max_seqlen, d))


def backward_varlen(q, k, v, o, lse, do, cu_seqlens, max_seqlen, causal=False, window=None,
                    scale=None, workspace=None, dq=None, dk=None, dv=None, stream=None,
                    dropout=None):
    """dQ, dK, dV [total,H,d] of packed sequences; see ``fa_backward_varlen``."""
    lib = load()
    _check_packed(q, k, v, o, do)
    B = _check_cu(cu_seqlens)
    total, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = varlen_workspace_bytes(B, H, total, int(max_seqlen), d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    m = _mask(1, causal, None, None, 0, window, dropout)
    st = lib.fa_backward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens), B, H, total,
                                int(max_seqlen), d, scale, ctypes.byref(m), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_backward_varlen")
    return dq, dk, dv


def fp8_workspace_bytes(B, H, N, d):
    return int(load().fa_fp8_workspace_bytes(B, H, N, d))


def fp8_workspace_views(ws, B, H, N):
    """Views of the parts of an FP8 workspace (layout in include/fa_fp8.h):
    q8, k8 uint8 [B*H, N, 128], vt8 uint8 [B*H, 128, Np], q/k scales fp32
    [B*H, T], v scales fp32 [B*H]."""
    T = (N + 127) // 128
    bh = B * H

    def r256(x):
        return -(-x // 256) * 256
    sizes = [bh * N * 128, bh * N * 128, bh * 128 * T * 128, bh * T * 4, bh * T * 4, bh * 4]
    offs = [0]
    for sz in sizes:
        offs.append(offs[-1] + r256(sz))
    u8 = ws.view(torch.uint8)
    q8 = u8[offs[0]:offs[0] + sizes[0]].view(bh, N, 128)
    k8 = u8[offs[1]:offs[1] + sizes[1]].view(bh, N, 128)
    vt8 = u8[offs[2]:offs[2] + sizes[2]].view(bh, 128, T * 128)
    qs = u8[offs[3]:offs[3] + sizes[3]].view(torch.float32).view(bh, T)
    ks = u8[offs[4]:offs[4] + sizes[4]].view(torch.float32).view(bh, T)
    vs = u8[offs[5]:offs[5] + sizes[5]].view(torch.float32)
    return dict(q8=q8, k8=k8, vt8=vt8, qs=qs, ks=ks, vs=vs)


def fp8_quantize(q, k, v, workspace=None, stream=None):
    """Block-quantise bf16 q, k, v [B,H,N,128] to e4m3 into a workspace
    (``fa_fp8_quantize``); returns the workspace."""
    lib = load()
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    nbytes = fp8_workspace_bytes(B, H, N, d)
    if nbytes == 0:
        raise FAError(FA_ERR_UNSUPPORTED if d != 128 else FA_ERR_INVALID_ARG, "fa_fp8_quantize")
    if workspace is None:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    st = lib.fa_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fp8_quantize")
    return workspace


def forward_fp8(q, k, v, causal=False, scale=None, workspace=None, out=None, lse=None,
                stream=None):
    """O, LSE of the FP8 forward with block quantisation (include/fa_fp8.h);
    q, k, v bf16 [B,H,N,128]."""
    lib = load()
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = fp8_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32) if lse is None else lse
    st = lib.fa_forward_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, scale,
                            int(bool(causal)), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_forward_fp8")
    return out, lse


def kvcache_num_splits(B, H, Nq, Nk, d, num_sms=0):
    """Split count ``forward_kvcache`` picks with ``num_splits=0``."""
    return int(load().fa_kvcache_num_splits(B, H, Nq, Nk, d, num_sms))


def kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits=0):
    return int(load().fa_kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits))


def forward_kvcache(q, k_cache, v_cache, cache_len=None, causal=False, scale=None,
                    num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """O, LSE of q [B,H,Nq,d] against a [B,H,Nk,d] key/value cache whose
    first cache_len[b] slots are valid; see include/fa_kvcache.h."""
    lib = load()
    for t in (q, k_cache, v_cache):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
            raise ValueError("q, k_cache, v_cache must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k_cache.shape[2]
    if tuple(k_cache.shape) != (B, H, Nk, d) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must be [B, H, Nk, d] with q's B, H, d")
    if cache_len is not None and not (cache_len.is_cuda and cache_len.dtype == torch.int32
                                      and cache_len.is_contiguous()
                                      and tuple(cache_len.shape) == (B,)):
        raise ValueError(f"cache_len must be a contiguous int32 CUDA [{B}] tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if num_splits == 0:
        num_splits = kvcache_num_splits(B, H, Nq, Nk, d)
    nbytes = kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32) if lse is None else lse
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.fa_forward_kvcache(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse),
                                B, H, Nq, Nk, d, scale, int(bool(causal)), _ptr(cache_len),
                                int(num_splits), _ptr(workspace), wsb, _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_forward_kvcache")
    return out, lse


def combine(o_parts, lse_parts, out=None, lse=None, stream=None):
    """Merge partial results over disjoint key sets: o_parts fp32 [S, rows, d]
    (normalised), lse_parts fp32 [S, rows] -> (O bf16 [rows, d], LSE fp32
    [rows]); see ``fa_combine``."""
    lib = load()
    if not (o_parts.is_cuda and o_parts.dtype == torch.float32 and o_parts.is_contiguous()
            and o_parts.dim() == 3):
        raise ValueError("o_parts must be a contiguous fp32 CUDA [S, rows, d] tensor")
    S, rows, d = o_parts.shape
    if not (lse_parts.is_cuda and lse_parts.dtype == torch.float32
            and lse_parts.is_contiguous() and tuple(lse_parts.shape) == (S, rows)):
        raise ValueError(f"lse_parts must be a contiguous fp32 CUDA [{S}, {rows}] tensor")
    out = torch.empty((rows, d), device=o_parts.device, dtype=torch.bfloat16) if out is None else out
    lse = torch.empty(rows, device=o_parts.device, dtype=torch.float32) if lse is None else lse
    st = lib.fa_combine(_ptr(o_parts), _ptr(lse_parts), S, rows, d, _ptr(out), _ptr(lse),
                        _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_combine")
    return out, lse


def tile_schedule(N, causal=False, block_mask=None, kv_len=None, b=0, device="cuda",
                  window=None):
    """(row_ptr, col_idx, partial) CUDA tensors; see ``fa_tile_schedule_masked``."""
    lib = load()
    T = (N + 127) // 128
    B = 0 if kv_len is None else kv_len.shape[0]
    m = _mask(N, causal, block_mask, kv_len, B, window)
    row_ptr = torch.zeros(T + 1, device=device, dtype=torch.int32)
    col_idx = torch.full((T * T,), -1, device=device, dtype=torch.int32)
    partial = torch.full((T * T,), 255, device=device, dtype=torch.uint8)
    st = lib.fa_tile_schedule_masked(N, ctypes.byref(m), b, _ptr(row_ptr),
                                     _ptr(col_idx), _ptr(partial), _stream())
    if st != FA_OK:
        raise FAError(st, "fa_tile_schedule_masked")
    return row_ptr, col_idx, partial


def last_device_status(stream=None):
    return int(load().fa_last_device_status(_stream(stream)))


def selftest_mma(mode, a, b, n=128, stream=None):
    """Single-tile tensor-core self-test (include/fa_selftest.h); returns c."""
    lib = load()
    rows = 128
    cols = 128 if mode == 0 else n
    c = torch.full((rows, cols), float("nan"), device=a.device, dtype=torch.float32)
    st = lib.fa_selftest_mma(int(mode), _ptr(a), _ptr(b), _ptr(c), int(n), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_selftest_mma")
    return c
