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


def bf16_storage_excess(got, ref):
    """Largest |got - ref| left after allowing each element the bf16 rounding
    of its own stored value.  A bf16 output holds round(v) of the kernel's
    fp32 result v, at most half a bf16 ulp of the element away from it; so
    |got - ref| - halfulp(got) <= |v - ref|, the arithmetic error that the
    tolerance is about.  (Comparing against round(ref) instead would count a
    whole ulp whenever v and ref fall on opposite sides of a rounding
    boundary, which at |x| in [4, 8) is 2^-5 = 0.031 for any tiny error.)"""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.maximum(np.abs(got), np.abs(ref))
    with np.errstate(divide="ignore"):
        expo = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    half_ulp = np.where(mag > 0, np.exp2(expo - 8.0), 0.0)  # bf16: 8 significant bits
    return float(np.max(np.abs(got - ref) - half_ulp)) if got.size else 0.0


def grad_sum_errors(dv, dk, do_pos, q_pos, pos_of_row, G: int = 1):
    """Worst ratio (error / bound) over every (b, h, column) of the two
    gradient invariants of causal softmax attention, on full GPU tensors:
        sum_t dV_t = sum_p dO_p   (every row of P sums to 1)
        sum_t dK_t = 0            (every row of dS sums to 0).
    dv, dk: [B, Hkv, S, D] device tensors in layout row order; pos_of_row:
    int64 [S] device tensor, the position each row holds; do_pos, q_pos:
    [B, H, S, D] inputs in POSITION order (device tensors); G = H / Hkv
    query heads share a key/value head (their sums add up).
    Bound per column c (fp64 sums, so the sums add no error of their own):
      4 * 2^-9 * ( sqrt(sum_t x_tc^2) + sqrt(sum_p y_pc^2 * w_p) )
        + 2^-24 * sum_t n_t |x_tc|  + 1e-3
    * storage: each stored bf16 value is off by at most half an ulp
      (<= 2^-8 relative, unbiased), so the sum of S of them has a standard
      deviation below 2^-9 sqrt(sum x^2); 4 of those.
    * operands: P (and dS) are rounded to bf16 as tensor-core operands, so
      row p's weights sum to 1 only up to about 2^-9 sqrt(sum_t P_pt^2); for
      these inputs (N(0,1) q, k at scale 1/sqrt(D): scores ~ N(0,1)) a row of
      p+1 kept keys has sum_t P_pt^2 ~ e/(p+1) =: w_p.  The row errors enter
      the dV sum weighted by dO_p and the dK sum by scale * |dP| * q_p ~ q_p
      (|dP| ~ sqrt(D) for unit dO, v).
    * accumulation: the dV/dK accumulator of key row t (key position s_t) is
      summed in the tensor core's fp32 over n_t = G (S - s_t) / 16 MMA steps
      (one step per 16 queries), and each step can lose up to an ulp of the
      running sum (the tensor core does not round the accumulation to
      nearest), half an ulp on average: a bias of up to 2^-24 n_t |x_t|
      toward zero, the same sign for every step, so it adds up over the
      column instead of averaging out.
    Returns {"dv"|"dk": (max error, smallest bound, max error/bound)} and,
    under "dv_shrink", the least-squares factor delta in
    sum_t dV_t = (1 - delta) sum_p dO_p over all columns with its
    correlation (a systematic shrink shows as delta > 0, corr near 1)."""
    import torch

    B, Hkv, S, D = dv.shape
    pos = torch.arange(S, device=do_pos.device, dtype=torch.float64)
    w = torch.clamp(np.e / (pos + 1.0), max=1.0).view(S, 1)
    n_row = (G * (S - pos_of_row.to(torch.float64)) / 16.0).view(S, 1)
    out = {}
    for name, x, y, has_target in (("dv", dv, do_pos, True), ("dk", dk, q_pos, False)):
        sx = x.double().sum(2)
        if has_target:
            want = y.double().sum(2).reshape(B, Hkv, G, D).sum(2)
        else:
            want = torch.zeros_like(sx)
        diff = sx - want
        err = diff.abs()
        x2 = torch.zeros_like(sx)
        y2 = torch.zeros_like(sx)
        acc = torch.zeros_like(sx)
        for h in range(Hkv):  # per head keeps the fp64 temporaries small
            xh = x[:, h].double()
            x2[:, h] = xh.square().sum(1)
            acc[:, h] = (xh.abs() * n_row).sum(1)
            for g in range(G):
                y2[:, h] += (y[:, h * G + g].double().square() * w).sum(1)
        bound = 4.0 * 2.0 ** -9 * (x2.sqrt() + y2.sqrt()) + 2.0 ** -24 * acc + 1e-3
        out[name] = (float(err.max()), float(bound.min()), float((err / bound).max()))
        if has_target:
            a, b_ = -diff.flatten(), want.flatten()
            delta = float((a * b_).sum() / (b_ * b_).sum())
            corr = float((a * b_).sum() / ((a * a).sum().sqrt() * (b_ * b_).sum().sqrt()))
            out["dv_shrink"] = (delta, corr)
    return out
