"""Shared helpers of the GPU parity tests (layout mapping, error metrics)."""
import numpy as np
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs

TOL = {torch.float32: {"o": 1e-4, "lse": 1e-4, "grad": 1e-4},
       torch.bfloat16: {"o": 2e-2, "lse": 1e-3, "grad": 2e-2}}


def positions(S, N, layout):
    """pos[row] = sequence position held by layout row (from the oracle)."""
    return oracle.layout_positions(S, N, layout)


def to_layout(x_cpu, N, layout, dev):
    """Position-order CPU tensor -> device tensor in the layout's row order
    (the GPU permute kernel does the striping)."""
    xd = x_cpu.to(dev).contiguous()
    if layout == sp.STRIPED:
        return sp.striped_permute(xd, N)
    if layout == sp.ZIGZAG:
        return sp.layout_permute(xd, N, sp.ZIGZAG)
    return xd


def to_positions(t_gpu, N, layout):
    """Device tensor in layout row order -> float64 numpy in position order
    (row r holds position pos[r]; mapped on the host)."""
    t = t_gpu.float().cpu().numpy().astype(np.float64)
    S = t.shape[2]
    pos = positions(S, N, layout)
    out = np.empty_like(t)
    out[:, :, pos] = t
    return out


def inputs(B, H, S, D, dtype, seed=0, with_do=True):
    return attention_inputs(B, H, S, D, dtype, seed=seed, with_do=with_do)


def head64(x, b, h):
    return x[b, h].double().numpy()


def maxerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def with_bf16_storage(tol, ref):
    """Bound for a bf16-stored output in cases beyond the benchmark
    workloads: the arithmetic bound `tol` plus the bf16 storage rounding of
    the largest value, 2^-8 of its magnitude (half the 2^-7 relative spacing
    of bf16 numbers).  At |ref| ~ 5 the storage alone can cost 0.016."""
    return tol + 2.0 ** -8 * float(np.max(np.abs(ref)))
