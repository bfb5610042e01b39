"""Python binding of libstriped -- striped causal attention on one GB300.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libstriped.so`` (built in-tree by :mod:`.build`).  PyTorch provides device
memory and the current stream; nothing here computes attention.  If the
library is missing, every call raises -- there is no fallback.

The functions mirror the C ABI in ``include/striped.h`` (same names).  Tensors
are CUDA tensors [B, H, S, D], contiguous, bf16 or fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

STRIPED = 0
CONTIGUOUS = 1
ZIGZAG = 2
BF16 = 0
FP32 = 1
FAULT_NONE = 0
FAULT_FWD_SKIP_KV = 1
FAULT_BWD_SKIP_Q = 2

_STATUS = {
    0: "ok", -1: "invalid argument", -2: "unsupported configuration", -3: "misaligned",
    -4: "CUDA error", -5: "device wait timed out", -6: "workspace missing or too small",
}

_lock = threading.Lock()
_lib = None


class StripedError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = ""
        if status == -4 and _lib is not None:
            extra = f" (cudaError {_lib.striped_last_cuda_error()})"
        super().__init__(f"{where}: {_STATUS.get(status, status)}{extra}")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libstriped.so (building it first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libstriped.so not built ({path}); run __graft_entry__.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        P, I64, I, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.striped_permute.argtypes = [P, P, I64, I64, I64, I64, I, I, P]
        lib.striped_unpermute.argtypes = [P, P, I64, I64, I64, I64, I, I, P]
        lib.striped_layout_permute.argtypes = [P, P, I64, I64, I64, I64, I, I, I, P]
        lib.striped_layout_unpermute.argtypes = [P, P, I64, I64, I64, I64, I, I, I, P]
        lib.striped_attn_fwd.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I, I, I, F, P, P]
        lib.striped_attn_fwd_gqa.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I, I, I, F, P, P]
        lib.striped_workspace_size.argtypes = [I64, I64, I64, I64, I, I]
        lib.striped_workspace_size.restype = SZ
        lib.striped_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I64, I64, I64, I64, I, I, I, F,
                                         P, P]
        lib.striped_attn_bwd_gqa.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I64, I64, I64, I64, I64, I, I, I,
                                             F, P, P]
        lib.ring_round_fwd.argtypes = [P, P, P, P, P, P, I, I, I64, I64, I64, I64, I, I64, I64, I, I, F, I,
                                       P, P]
        lib.ring_bwd_workspace_size.argtypes = [I64, I64, I64, I64, I]
        lib.ring_bwd_workspace_size.restype = SZ
        lib.ring_bwd_prepare.argtypes = [P, P, P, P, SZ, P, I64, I64, I64, I64, I, P]
        lib.ring_round_bwd.argtypes = [P, P, P, P, P, SZ, P, P, P, I, I, I64, I64, I64, I64, I, I, I, F, I, P, P]
        lib.ring_bwd_finish.argtypes = [P, P, I64, I, F, P]
        lib.striped_varlen_permute.argtypes = [P, P, P, I, I64, I64, I, I, I, P]
        lib.striped_varlen_unpermute.argtypes = [P, P, P, I, I64, I64, I, I, I, P]
        lib.striped_attn_fwd_varlen.argtypes = [P, P, P, P, P, P, I, I64, I64, I64, I, I, I, F, P, P]
        lib.striped_attn_bwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, P, I, I64, I64, I64, I, I, I,
                                                F, P, P]
        lib.striped_kernel_tile.argtypes = [I, I64, P, P]
        lib.striped_fwd_query_tiles_per_cta.argtypes = [I64, I64, I64, I64, I, I, I, I]
        lib.striped_tile_counts.argtypes = [I64, I, I, I, I, P, P]
        lib.striped_critical_path.argtypes = [I64, I, I, I, I]
        lib.striped_critical_path.restype = I64
        lib.striped_tile_counts_varlen.argtypes = [P, I, I, I, I, I, P, P]
        lib.striped_critical_path_varlen.argtypes = [P, I, I, I, I, I]
        lib.striped_critical_path_varlen.restype = I64
        lib.striped_check_error.argtypes = [P]
        lib.striped_status_string.argtypes = [I]
        lib.striped_status_string.restype = ctypes.c_char_p
        lib.striped_last_cuda_error.argtypes = []
        lib.striped_selftest_timeout.argtypes = [I64, P]
        lib.striped_test_inject.argtypes = [I, I64]
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise StripedError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr_or_null(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------------ permute
def striped_permute(x: torch.Tensor, N: int, out: torch.Tensor | None = None, stream=None):
    """Row d*L+i of the result holds position i*N+d of x ([B,H,S,D])."""
    B, H, S, D = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(load().striped_permute(_dev(x, "x"), _dev(y, "y"), B, H, S, D, N, _dtype_code(x),
                                  _stream(stream)), "striped_permute")
    return y


def striped_unpermute(x: torch.Tensor, N: int, out: torch.Tensor | None = None, stream=None):
    """Inverse of striped_permute."""
    B, H, S, D = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(load().striped_unpermute(_dev(x, "x"), _dev(y, "y"), B, H, S, D, N, _dtype_code(x),
                                    _stream(stream)), "striped_unpermute")
    return y


def layout_permute(x: torch.Tensor, N: int, layout: int, out: torch.Tensor | None = None, stream=None):
    """Position order -> `layout` row order (striped, contiguous or zig-zag)."""
    B, H, S, D = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(load().striped_layout_permute(_dev(x, "x"), _dev(y, "y"), B, H, S, D, N, layout, _dtype_code(x),
                                         _stream(stream)), "striped_layout_permute")
    return y


def layout_unpermute(x: torch.Tensor, N: int, layout: int, out: torch.Tensor | None = None, stream=None):
    """Inverse of layout_permute."""
    B, H, S, D = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(load().striped_layout_unpermute(_dev(x, "x"), _dev(y, "y"), B, H, S, D, N, layout,
                                           _dtype_code(x), _stream(stream)), "striped_layout_unpermute")
    return y


# ------------------------------------------------------------------ attention
def kernel_tile(dtype: torch.dtype, D: int) -> int:
    tq, tk = ctypes.c_int(), ctypes.c_int()
    code = BF16 if dtype == torch.bfloat16 else FP32
    _check(load().striped_kernel_tile(code, D, ctypes.byref(tq), ctypes.byref(tk)), "striped_kernel_tile")
    return tq.value


def fwd_query_tiles_per_cta(B: int, H: int, S: int, D: int, N: int, layout: int = STRIPED,
                            dtype: torch.dtype = torch.bfloat16, num_sms: int | None = None) -> int:
    """Query tiles one forward CTA runs (1, or 2 for the stripe-pair
    schedule) on a GPU with num_sms multiprocessors (default: the current
    CUDA device's)."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    code = BF16 if dtype == torch.bfloat16 else FP32
    r = load().striped_fwd_query_tiles_per_cta(B, H, S, D, N, layout, code, num_sms)
    if r < 0:
        raise StripedError(r, "striped_fwd_query_tiles_per_cta")
    return r


def new_tile_stats(N: int, device) -> torch.Tensor:
    """Zeroed int64 [2, N, N] device counter array for tile_stats."""
    return torch.zeros((2, N, N), dtype=torch.int64, device=device)


def striped_attn_fwd(q, k, v, N: int, layout: int = STRIPED, scale: float | None = None,
                     tile_stats: torch.Tensor | None = None, out=None, lse_out=None, stream=None):
    """Causal attention of all N ring rounds; returns (o, lse).  k and v may
    have fewer heads than q (grouped-query attention, striped_attn_fwd_gqa)."""
    if k.shape[1] != q.shape[1]:
        return striped_attn_fwd_gqa(q, k, v, N, layout, scale, tile_stats, out, lse_out, stream)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / D ** 0.5
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse_out is None else lse_out
    _check(load().striped_attn_fwd(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"), _dev(lse, "lse"),
                                   B, H, S, D, N, layout, _dtype_code(q), float(scale),
                                   _ptr_or_null(tile_stats), _stream(stream)), "striped_attn_fwd")
    return o, lse


def striped_attn_fwd_gqa(q, k, v, N: int, layout: int = STRIPED, scale: float | None = None,
                         tile_stats: torch.Tensor | None = None, out=None, lse_out=None, stream=None):
    """Grouped-query form: q [B,H,S,D], k and v [B,Hkv,S,D] (H % Hkv == 0);
    query head h reads key/value head h // (H/Hkv).  Returns (o, lse)."""
    B, H, S, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / D ** 0.5
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse_out is None else lse_out
    _check(load().striped_attn_fwd_gqa(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"),
                                       _dev(lse, "lse"), B, H, Hkv, S, D, N, layout, _dtype_code(q),
                                       float(scale), _ptr_or_null(tile_stats), _stream(stream)),
           "striped_attn_fwd_gqa")
    return o, lse


def workspace_size(B: int, H: int, S: int, D: int, N: int, dtype: torch.dtype) -> int:
    code = BF16 if dtype == torch.bfloat16 else FP32
    return int(load().striped_workspace_size(B, H, S, D, N, code))


def new_workspace(B, H, S, D, N, dtype, device) -> torch.Tensor:
    n = workspace_size(B, H, S, D, N, dtype)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def striped_attn_bwd(q, k, v, o, lse, dO, N: int, layout: int = STRIPED, scale: float | None = None,
                     workspace: torch.Tensor | None = None, tile_stats: torch.Tensor | None = None,
                     dq=None, dk=None, dv=None, stream=None):
    """Backward of striped_attn_fwd; returns (dq, dk, dv).  k and v may have
    fewer heads than q (grouped-query attention, striped_attn_bwd_gqa)."""
    B, H, S, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / D ** 0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = new_workspace(B, H, S, D, N, q.dtype, q.device) if workspace is None else workspace
    args = [_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"), _dev(lse, "lse"), _dev(dO, "dO"),
            _dev(dq, "dq"), _dev(dk, "dk"), _dev(dv, "dv"), _dev(ws, "workspace"),
            ws.numel() * ws.element_size()]
    tail = [S, D, N, layout, _dtype_code(q), float(scale), _ptr_or_null(tile_stats), _stream(stream)]
    if Hkv != H:
        _check(load().striped_attn_bwd_gqa(*args, B, H, Hkv, *tail), "striped_attn_bwd_gqa")
    else:
        _check(load().striped_attn_bwd(*args, B, H, *tail), "striped_attn_bwd")
    return dq, dk, dv


striped_attn_bwd_gqa = striped_attn_bwd  # same call; k, v (and dk, dv) carry Hkv heads


def ring_round_fwd(q, k, v, o_acc, lse_acc, d: int, e: int, N: int, layout: int = STRIPED,
                   scale: float | None = None, first_round: bool = False, o_out=None,
                   tile_stats: torch.Tensor | None = None, stream=None):
    """One ring round of virtual device d against key stripe e, merged into
    (o_acc fp32 [B,H,S,D], lse_acc fp32 [B,H,S]).  q, k, v are the FULL
    [B,H,S,D] tensors; the stripe slices are taken here by pointer offset
    (a "send to the next device" is a pointer to the next stripe)."""
    B, H, S, D = q.shape
    L = S // N
    if scale is None:
        scale = 1.0 / D ** 0.5
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o_acc, "o_acc"), (lse_acc, "lse_acc")):
        _dev(t, nm)
    if o_acc.dtype != torch.float32 or lse_acc.dtype != torch.float32:
        raise TypeError("o_acc and lse_acc must be fp32")
    es = q.element_size()
    qd = ctypes.c_void_p(q.data_ptr() + d * L * D * es)
    ke = ctypes.c_void_p(k.data_ptr() + e * L * D * es)
    ve = ctypes.c_void_p(v.data_ptr() + e * L * D * es)
    oa = ctypes.c_void_p(o_acc.data_ptr() + d * L * D * 4)
    la = ctypes.c_void_p(lse_acc.data_ptr() + d * L * 4)
    oo = None if o_out is None else ctypes.c_void_p(_dev(o_out, "o_out").value + d * L * D * es)
    _check(load().ring_round_fwd(qd, ke, ve, oa, la, oo, d, e, B, H, L, D, N, S * D, S, layout,
                                 _dtype_code(q), float(scale), 1 if first_round else 0,
                                 _ptr_or_null(tile_stats), _stream(stream)), "ring_round_fwd")


# ------------------------------------------------------------------ one device of a ring
def ring_bwd_workspace(q_d: torch.Tensor) -> torch.Tensor:
    """Statistics workspace of ring_bwd_prepare / ring_round_bwd for a
    device's block q_d [B, H, L, D] (bf16)."""
    B, H, L, D = q_d.shape
    n = int(load().ring_bwd_workspace_size(B, H, L, D, _dtype_code(q_d)))
    if n == 0:
        raise StripedError(-1, "ring_bwd_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=q_d.device)


def ring_bwd_prepare(o_d, lse_d, dO_d, workspace, dq_acc, stream=None):
    """Statistics of device d's query block into workspace; zero dq_acc."""
    B, H, L, D = o_d.shape
    _check(load().ring_bwd_prepare(_dev(o_d, "o_d"), _dev(lse_d, "lse_d"), _dev(dO_d, "dO_d"),
                                   _dev(workspace, "workspace"), workspace.numel(), _dev(dq_acc, "dq_acc"),
                                   B, H, L, D, _dtype_code(o_d), _stream(stream)), "ring_bwd_prepare")


def ring_round_bwd(q_d, k_e, v_e, dO_d, workspace, dq_acc, dk_acc, dv_acc, d: int, e: int, N: int,
                   layout: int = STRIPED, scale: float | None = None, first_round: bool = False,
                   tile_stats: torch.Tensor | None = None, stream=None):
    """Device d's backward round against key/value block e: dQ share into
    dq_acc, dK/dV shares into (or, first_round, onto) dk_acc/dv_acc (fp32
    [B, H, L, D] sums travelling with block e)."""
    B, H, L, D = q_d.shape
    if scale is None:
        scale = 1.0 / D ** 0.5
    for t, nm in ((dq_acc, "dq_acc"), (dk_acc, "dk_acc"), (dv_acc, "dv_acc")):
        if t.dtype != torch.float32:
            raise TypeError(f"{nm} must be fp32")
    _check(load().ring_round_bwd(_dev(q_d, "q_d"), _dev(k_e, "k_e"), _dev(v_e, "v_e"), _dev(dO_d, "dO_d"),
                                 _dev(workspace, "workspace"), workspace.numel(), _dev(dq_acc, "dq_acc"),
                                 _dev(dk_acc, "dk_acc"), _dev(dv_acc, "dv_acc"), d, e, B, H, L, D, N, layout,
                                 _dtype_code(q_d), float(scale), 1 if first_round else 0, _ptr_or_null(tile_stats),
                                 _stream(stream)), "ring_round_bwd")


def ring_bwd_finish(acc: torch.Tensor, mul: float, out: torch.Tensor | None = None, stream=None):
    """out = bf16(mul * acc) (the final dQ with mul = scale, dK / dV with 1)."""
    y = torch.empty(acc.shape, dtype=torch.bfloat16, device=acc.device) if out is None else out
    _check(load().ring_bwd_finish(_dev(acc, "acc"), _dev(y, "out"), acc.numel(), BF16, float(mul),
                                  _stream(stream)), "ring_bwd_finish")
    return y


def ring_round_fwd_block(q_d, k_e, v_e, o_acc, lse_acc, d: int, e: int, N: int, layout: int = STRIPED,
                         scale: float | None = None, first_round: bool = False, o_out=None,
                         tile_stats: torch.Tensor | None = None, stream=None):
    """ring_round_fwd on one device's own contiguous blocks ([B, H, L, D]
    tensors; o_acc fp32 of the same shape, lse_acc fp32 [B, H, L])."""
    B, H, L, D = q_d.shape
    if scale is None:
        scale = 1.0 / D ** 0.5
    if o_acc.dtype != torch.float32 or lse_acc.dtype != torch.float32:
        raise TypeError("o_acc and lse_acc must be fp32")
    oo = None if o_out is None else _dev(o_out, "o_out")
    _check(load().ring_round_fwd(_dev(q_d, "q_d"), _dev(k_e, "k_e"), _dev(v_e, "v_e"), _dev(o_acc, "o_acc"),
                                 _dev(lse_acc, "lse_acc"), oo, d, e, B, H, L, D, N, L * D, L, layout,
                                 _dtype_code(q_d), float(scale), 1 if first_round else 0,
                                 _ptr_or_null(tile_stats), _stream(stream)), "ring_round_fwd")


# ------------------------------------------------------------------ packed sequences
def _cu_host(cu_seqlens):
    """cu_seqlens (list, numpy or CPU tensor) -> contiguous host int32 array."""
    import numpy as np

    if isinstance(cu_seqlens, torch.Tensor):
        cu_seqlens = cu_seqlens.cpu().numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return cu, cu.ctypes.data_as(ctypes.c_void_p), len(cu) - 1


def striped_varlen_permute(x: torch.Tensor, cu_seqlens, N: int, layout: int = STRIPED, out=None, stream=None):
    """Packed head [H, S, D] in position order -> each sequence placed on
    its own, device slices of all sequences concatenated."""
    H, S, D = x.shape
    y = torch.empty_like(x) if out is None else out
    cu, cp, n = _cu_host(cu_seqlens)
    _check(load().striped_varlen_permute(_dev(x, "x"), _dev(y, "y"), cp, n, H, D, N, layout, _dtype_code(x),
                                         _stream(stream)), "striped_varlen_permute")
    return y


def striped_varlen_unpermute(x: torch.Tensor, cu_seqlens, N: int, layout: int = STRIPED, out=None, stream=None):
    """Inverse of striped_varlen_permute."""
    H, S, D = x.shape
    y = torch.empty_like(x) if out is None else out
    cu, cp, n = _cu_host(cu_seqlens)
    _check(load().striped_varlen_unpermute(_dev(x, "x"), _dev(y, "y"), cp, n, H, D, N, layout, _dtype_code(x),
                                           _stream(stream)), "striped_varlen_unpermute")
    return y


def striped_attn_fwd_varlen(q, k, v, cu_seqlens, N: int, layout: int = STRIPED, scale: float | None = None,
                            tile_stats: torch.Tensor | None = None, out=None, lse_out=None, stream=None):
    """Packed sequences: q [H,S,D], k and v [Hkv,S,D]; returns (o, lse [H,S])."""
    H, S, D = q.shape
    Hkv = k.shape[0]
    if scale is None:
        scale = 1.0 / D ** 0.5
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, S), dtype=torch.float32, device=q.device) if lse_out is None else lse_out
    cu, cp, n = _cu_host(cu_seqlens)
    _check(load().striped_attn_fwd_varlen(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"),
                                          _dev(lse, "lse"), cp, n, H, Hkv, D, N, layout, _dtype_code(q),
                                          float(scale), _ptr_or_null(tile_stats), _stream(stream)),
           "striped_attn_fwd_varlen")
    return o, lse


def striped_attn_bwd_varlen(q, k, v, o, lse, dO, cu_seqlens, N: int, layout: int = STRIPED,
                            scale: float | None = None, workspace=None, tile_stats=None, dq=None, dk=None, dv=None,
                            stream=None):
    """Backward of striped_attn_fwd_varlen; returns (dq, dk, dv)."""
    H, S, D = q.shape
    Hkv = k.shape[0]
    if scale is None:
        scale = 1.0 / D ** 0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = new_workspace(1, H, S, D, N, q.dtype, q.device) if workspace is None else workspace
    cu, cp, n = _cu_host(cu_seqlens)
    _check(load().striped_attn_bwd_varlen(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"),
                                          _dev(lse, "lse"), _dev(dO, "dO"), _dev(dq, "dq"), _dev(dk, "dk"),
                                          _dev(dv, "dv"), _dev(ws, "workspace"), ws.numel() * ws.element_size(),
                                          cp, n, H, Hkv, D, N, layout, _dtype_code(q), float(scale),
                                          _ptr_or_null(tile_stats), _stream(stream)), "striped_attn_bwd_varlen")
    return dq, dk, dv


# ------------------------------------------------------------------ host model
def tile_counts(S: int, N: int, Tq: int, Tk: int, layout: int = STRIPED):
    """(full, partial) int64 numpy tables [N rounds, N devices] per (b, h)."""
    import numpy as np

    full = np.zeros(N * N, dtype=np.int64)
    part = np.zeros(N * N, dtype=np.int64)
    _check(load().striped_tile_counts(S, N, Tq, Tk, layout, full.ctypes.data_as(ctypes.c_void_p),
                                      part.ctypes.data_as(ctypes.c_void_p)), "striped_tile_counts")
    return full.reshape(N, N), part.reshape(N, N)


def critical_path(S: int, N: int, Tq: int, Tk: int, layout: int = STRIPED) -> int:
    r = int(load().striped_critical_path(S, N, Tq, Tk, layout))
    if r < 0:
        raise StripedError(r, "striped_critical_path")
    return r


def tile_counts_varlen(cu_seqlens, N: int, Tq: int, Tk: int, layout: int = STRIPED):
    """(full, partial) tables [N rounds, N devices] of a packed batch."""
    import numpy as np

    full = np.zeros(N * N, dtype=np.int64)
    part = np.zeros(N * N, dtype=np.int64)
    cu, cp, n = _cu_host(cu_seqlens)
    _check(load().striped_tile_counts_varlen(cp, n, N, Tq, Tk, layout, full.ctypes.data_as(ctypes.c_void_p),
                                             part.ctypes.data_as(ctypes.c_void_p)), "striped_tile_counts_varlen")
    return full.reshape(N, N), part.reshape(N, N)


def critical_path_varlen(cu_seqlens, N: int, Tq: int, Tk: int, layout: int = STRIPED) -> int:
    cu, cp, n = _cu_host(cu_seqlens)
    r = int(load().striped_critical_path_varlen(cp, n, N, Tq, Tk, layout))
    if r < 0:
        raise StripedError(r, "striped_critical_path_varlen")
    return r


def check_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().striped_check_error(_stream(stream)))


def selftest_timeout(spins: int, stream=None):
    _check(load().striped_selftest_timeout(int(spins), _stream(stream)), "striped_selftest_timeout")


def test_inject(fault: int, wait_limit_ns: int = 0):
    """TEST HOOK: make the kernels skip one of their loads (FAULT_*) and/or
    bound every device-side wait by wait_limit_ns (<= 0: the 2 s default)
    for every later launch on the current device; (FAULT_NONE, 0) restores."""
    _check(load().striped_test_inject(int(fault), int(wait_limit_ns)), "striped_test_inject")


def status_string(status: int) -> str:
    return load().striped_status_string(int(status)).decode()
