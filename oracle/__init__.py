"""Plain fp64 CPU oracle for striped causal attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, POSIX threads over
rows); this module compiles it with gcc on first use and wraps it with ctypes
over numpy float64 arrays.  Every function works on ONE head stored [S, D]
row-major in *position* (unpermuted) order.

Definitions followed (pages on "Striped Attention: Faster Ring Attention for
Causal Transformers"):

* exact causal attention -- research.elamur.ai summary page, §Summary and
  §Key points ("results remain exact"); pith.science paper page, abstract
  ("an exact attention algorithm");
* stripe placement "every N-th token" -- research.elamur.ai, §Summary;
* contiguous placement and per-round work of Ring Attention -- §Summary,
  first paragraph; per-round balance -- §Key points "Imbalance";
* the zig-zag placement (2N chunks, device d holds chunks d and 2N-1-d) is
  not on the pages: it is the usual load-balanced alternative, defined in
  ``oracle.c`` and compared against the striped placement;
* grouped-query attention (query head h reads key/value head h // G) is not
  on the pages either: ``attn_fwd_gqa`` / ``attn_bwd_gqa`` compose the
  per-head definition, summing the gradients of a shared key/value head;
* one ring round's share of the gradients (``bwd_block``): the pairs of one
  query block and one key block, with the rows' full-sequence LSE and
  Jacobian sums -- §Summary (blocks circulate, each device accumulates);
* packed variable-length batches (not on the pages): ``attn_fwd_varlen`` /
  ``attn_bwd_varlen`` apply the definition to each sequence on its own, and
  ``varlen_positions`` places each sequence on its own inside every device.

Pins: every function here is checked in ``tests/test_oracle.py`` against
things other than itself (closed forms, special cases, library routines,
finite differences, brute force).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

STRIPED = 0
CONTIGUOUS = 1
ZIGZAG = 2


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc -O2, no BLAS)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            Dbl = ctypes.c_double
            lib.oracle_position_of_row.argtypes = [I64, I64, I, I]
            lib.oracle_position_of_row.restype = I64
            lib.oracle_stripe_positions.argtypes = [I64, I, P]
            lib.oracle_zigzag_positions.argtypes = [I64, I, P]
            lib.oracle_attn_fwd.argtypes = [P, P, P, I64, I64, Dbl, P, I64, P, P, P, I]
            lib.oracle_bwd_rows.argtypes = [P, P, P, P, I64, I64, Dbl, P, I64, P, P, P, I]
            lib.oracle_bwd_keys.argtypes = [P, P, P, P, I64, I64, Dbl, P, P, I64, P, I64, P, P, I]
            lib.oracle_attn_bwd.argtypes = [P, P, P, P, I64, I64, Dbl, P, P, P, I]
            lib.oracle_bwd_block.argtypes = [P, P, P, P, P, I64, P, P, P, I64, I64, Dbl, P, P, P]
            lib.oracle_tile_counts_bruteforce.argtypes = [I64, I, I64, I64, I, P, P]
            lib.oracle_tile_counts_closed.argtypes = [I64, I, I64, I, P, P]
            lib.oracle_critical_path.argtypes = [P, P, I]
            lib.oracle_critical_path.restype = I64
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# placement
# --------------------------------------------------------------------------
def position_of_row(row: int, S: int, N: int, layout: int = STRIPED) -> int:
    """Global position held by layout row ``row`` (striped: d*L+i -> i*N+d)."""
    return int(_load().oracle_position_of_row(row, S, N, layout))


def stripe_positions(S: int, N: int) -> np.ndarray:
    """pos[row] for the striped layout, built by enumerating p mod N == d."""
    out = np.empty(S, dtype=np.int64)
    _load().oracle_stripe_positions(S, N, _ptr(out))
    return out


def zigzag_positions(S: int, N: int) -> np.ndarray:
    """pos[row] for the zig-zag layout, built by enumerating the positions
    whose chunk (of S/(2N)) is d or 2N-1-d."""
    out = np.empty(S, dtype=np.int64)
    _load().oracle_zigzag_positions(S, N, _ptr(out))
    return out


def layout_positions(S: int, N: int, layout: int) -> np.ndarray:
    """pos[row] of any layout (enumeration for striped and zig-zag)."""
    if layout == STRIPED:
        return stripe_positions(S, N)
    if layout == ZIGZAG:
        return zigzag_positions(S, N)
    return np.arange(S, dtype=np.int64)


# --------------------------------------------------------------------------
# forward / backward (one head, position order)
# --------------------------------------------------------------------------
def attn_fwd(q, k, v, scale: float, rows=None, key_in_set=None, nthreads: int | None = None):
    """Return (O [n, D], LSE [n]) for query positions ``rows`` (all if None).

    ``key_in_set`` (bool [S]) restricts the keys (one ring round's partial
    result); rows with no kept key get O = 0 and LSE = -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S, D = q.shape
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = S if r is None else r.shape[0]
    ks = None if key_in_set is None else np.ascontiguousarray(np.asarray(key_in_set, dtype=np.uint8))
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), S, D, float(scale), _ptr(r), n, _ptr(ks),
                            _ptr(o), _ptr(lse), nthreads or default_threads())
    return o, lse


def bwd_rows(q, k, v, dO, scale: float, rows=None, want_dq: bool = True,
             nthreads: int | None = None):
    """Return (LSE [n], J [n], dQ [n, D] or None) for query positions ``rows``."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    S, D = q.shape
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = S if r is None else r.shape[0]
    lse = np.empty(n, dtype=np.float64)
    J = np.empty(n, dtype=np.float64)
    dq = np.empty((n, D), dtype=np.float64) if want_dq else None
    _load().oracle_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), S, D, float(scale), _ptr(r), n,
                            _ptr(lse), _ptr(J), _ptr(dq), nthreads or default_threads())
    return lse, J, dq


def bwd_keys(q, k, v, dO, scale: float, keys, nthreads: int | None = None):
    """Return (dK [n, D], dV [n, D]) for key positions ``keys``.

    Computes the needed LSE_p and J_p for every query p >= min(keys) first.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    S, D = q.shape
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    nt = nthreads or default_threads()
    p_lo = int(keys.min()) if keys.size else S
    rows = np.arange(p_lo, S, dtype=np.int64)
    lse, J, _ = bwd_rows(q, k, v, dO, scale, rows=rows, want_dq=False, nthreads=nt)
    dk = np.empty((keys.shape[0], D), dtype=np.float64)
    dv = np.empty((keys.shape[0], D), dtype=np.float64)
    _load().oracle_bwd_keys(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), S, D, float(scale), _ptr(lse),
                            _ptr(J), p_lo, _ptr(keys), keys.shape[0], _ptr(dk), _ptr(dv), nt)
    return dk, dv


def attn_bwd(q, k, v, dO, scale: float, nthreads: int | None = None):
    """Full backward of one head: (dQ, dK, dV), each [S, D]."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    S, D = q.shape
    dq = np.empty((S, D), dtype=np.float64)
    dk = np.empty((S, D), dtype=np.float64)
    dv = np.empty((S, D), dtype=np.float64)
    _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), S, D, float(scale), _ptr(dq),
                            _ptr(dk), _ptr(dv), nthreads or default_threads())
    return dq, dk, dv


def bwd_block(q, dO, qpos, lse, J, k, v, kpos, scale: float):
    """One ring round's share of the gradients: query rows q, dO [nq, D] at
    positions qpos, key rows k, v [nk, D] at positions kpos, pairs with key
    position <= query position; lse, J are the query rows' full-sequence
    values.  Returns the partial (dq [nq, D], dk [nk, D], dv [nk, D])."""
    q, dO, k, v = _f64(q), _f64(dO), _f64(k), _f64(v)
    lse, J = _f64(lse), _f64(J)
    qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    kpos = np.ascontiguousarray(np.asarray(kpos, dtype=np.int64))
    nq, D = q.shape
    nk = k.shape[0]
    dq = np.empty((nq, D))
    dk = np.empty((nk, D))
    dv = np.empty((nk, D))
    _load().oracle_bwd_block(_ptr(q), _ptr(dO), _ptr(qpos), _ptr(lse), _ptr(J), nq, _ptr(k), _ptr(v), _ptr(kpos),
                             nk, D, float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


# --------------------------------------------------------------------------
# per-round tile accounting
# --------------------------------------------------------------------------
def tile_counts_bruteforce(S: int, N: int, Tq: int, Tk: int, layout: int = STRIPED):
    """(full [N rounds, N devices], partial [N, N]) by enumerating every pair."""
    full = np.zeros(N * N, dtype=np.int64)
    part = np.zeros(N * N, dtype=np.int64)
    _load().oracle_tile_counts_bruteforce(S, N, Tq, Tk, layout, _ptr(full), _ptr(part))
    return full.reshape(N, N), part.reshape(N, N)


def tile_counts_closed(S: int, N: int, T: int, layout: int = STRIPED):
    """Closed-form (full, partial) tables for T dividing L = S / N."""
    full = np.zeros(N * N, dtype=np.int64)
    part = np.zeros(N * N, dtype=np.int64)
    _load().oracle_tile_counts_closed(S, N, T, layout, _ptr(full), _ptr(part))
    return full.reshape(N, N), part.reshape(N, N)


def critical_path(full: np.ndarray, partial: np.ndarray) -> int:
    """Sum over rounds of the busiest device's tile count."""
    f = np.ascontiguousarray(full, dtype=np.int64)
    p = np.ascontiguousarray(partial, dtype=np.int64)
    return int(_load().oracle_critical_path(_ptr(f), _ptr(p), f.shape[0]))


# --------------------------------------------------------------------------
# grouped-query attention (not on the pages): H query heads share Hkv
# key/value heads, query head h reading key/value head h // (H / Hkv)
# --------------------------------------------------------------------------
def attn_fwd_gqa(q, k, v, scale: float, nthreads: int | None = None):
    """q [H, S, D], k and v [Hkv, S, D] (one batch entry) -> (O [H, S, D],
    LSE [H, S]): each query head is plain causal attention against its
    group's key/value head."""
    H, Hkv = q.shape[0], k.shape[0]
    G = H // Hkv
    outs = [attn_fwd(q[h], k[h // G], v[h // G], scale, nthreads=nthreads) for h in range(H)]
    return np.stack([o for o, _ in outs]), np.stack([l for _, l in outs])


def attn_bwd_gqa(q, k, v, dO, scale: float, nthreads: int | None = None):
    """Gradients of attn_fwd_gqa: dQ per query head; dK and dV of a shared
    key/value head are the sums of the gradients of every query head that
    reads it (the head is used G times)."""
    H, Hkv = q.shape[0], k.shape[0]
    G = H // Hkv
    dq = np.empty_like(np.asarray(q, dtype=np.float64))
    dk = np.zeros(np.shape(k), dtype=np.float64)
    dv = np.zeros(np.shape(v), dtype=np.float64)
    for h in range(H):
        gq, gk, gv = attn_bwd(q[h], k[h // G], v[h // G], dO[h], scale, nthreads=nthreads)
        dq[h] = gq
        dk[h // G] += gk
        dv[h // G] += gv
    return dq, dk, dv


# --------------------------------------------------------------------------
# packed variable-length batches (not on the pages): sequences
# [cu[i], cu[i+1]) of one packed head attend only within themselves
# --------------------------------------------------------------------------
def varlen_positions(cu_seqlens, N: int, layout: int) -> np.ndarray:
    """pos[row] of a packed head: device d's rows hold, sequence after
    sequence, that sequence's rows of device d under `layout` (each sequence
    placed on its own), so row d*L + cu[i]/N + j holds cu[i] + pos_i(d*L_i + j)
    with L = S/N and L_i = (cu[i+1] - cu[i]) / N."""
    cu = [int(c) for c in cu_seqlens]
    S = cu[-1]
    L = S // N
    pos = np.empty(S, dtype=np.int64)
    for i in range(len(cu) - 1):
        Si = cu[i + 1] - cu[i]
        Li = Si // N
        own = layout_positions(Si, N, layout)  # row -> position inside sequence i
        for d in range(N):
            pos[d * L + cu[i] // N: d * L + cu[i] // N + Li] = cu[i] + own[d * Li:(d + 1) * Li]
    return pos


def attn_fwd_varlen(q, k, v, cu_seqlens, scale: float, nthreads: int | None = None):
    """One packed head [S, D] in position order: causal attention inside each
    sequence, nothing across sequences (block-diagonal causal mask)."""
    cu = [int(c) for c in cu_seqlens]
    o = np.empty((cu[-1], np.shape(v)[1]))
    lse = np.empty(cu[-1])
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        o[a:b], lse[a:b] = attn_fwd(q[a:b], k[a:b], v[a:b], scale, nthreads=nthreads)
    return o, lse


def attn_bwd_varlen(q, k, v, dO, cu_seqlens, scale: float, nthreads: int | None = None):
    """Gradients of attn_fwd_varlen: each sequence's own backward."""
    cu = [int(c) for c in cu_seqlens]
    out = [np.empty((cu[-1], np.shape(q)[1])) for _ in range(3)]
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        g = attn_bwd(q[a:b], k[a:b], v[a:b], dO[a:b], scale, nthreads=nthreads)
        for t in range(3):
            out[t][a:b] = g[t]
    return tuple(out)


def merge_rounds(o_a, lse_a, o_b, lse_b):
    """Merge two normalised partial results (O, LSE) of disjoint key sets.

    The combination of per-round softmax partials is the log-sum-exp rule:
    lse = log(e^a + e^b); O = (e^a O_a + e^b O_b) / e^lse.  A side whose LSE
    is -inf (no kept key) contributes nothing.  Written in numpy here (fp64)
    because it is three lines; it is pinned in the tests by merging the
    per-round results of every stripe back into the full attention.
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    safe = np.where(np.isfinite(m), m, 0.0)
    wa = np.exp(lse_a - safe)
    wb = np.exp(lse_b - safe)
    w = wa + wb
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(np.isfinite(m), safe + np.log(w), -np.inf)
        o = np.where(np.isfinite(m)[:, None],
                     (wa[:, None] * o_a + wb[:, None] * o_b) / np.where(w > 0, w, 1.0)[:, None],
                     o_a)
    return o, lse
