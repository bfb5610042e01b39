"""Backward parity on the GPU against the fp64 oracle (direct
differentiation with the softmax-Jacobian row sum, which shares no code path
with the kernels' Delta = <dO, O> form), tile counters, and the gradient
invariants sum_t dV_t = sum_p dO_p and sum_t dK_t = 0."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from tests._util import TOL, grad_sum_errors, head64, inputs, maxerr, to_layout, to_positions

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run(B, H, S, D, N, layout, dtype, seed=0):
    x = inputs(B, H, S, D, dtype, seed=seed)
    q, k, v, do = (to_layout(x[n], N, layout, DEV) for n in ("q", "k", "v", "do"))
    o, lse = sp.striped_attn_fwd(q, k, v, N, layout)
    stats = sp.new_tile_stats(N, DEV)
    dq, dk, dv = sp.striped_attn_bwd(q, k, v, o, lse, do, N, layout, tile_stats=stats)
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    return x, (dq, dk, dv), stats


def _check(x, grads, stats, B, H, S, D, N, layout, dtype, heads=None):
    scale = 1.0 / D ** 0.5
    got = [to_positions(t, N, layout) for t in grads]
    tol = TOL[dtype]["grad"]
    worst = [0.0, 0.0, 0.0]
    for b in range(B):
        for h in (range(H) if heads is None else heads):
            ref = oracle.attn_bwd(head64(x["q"], b, h), head64(x["k"], b, h), head64(x["v"], b, h),
                                  head64(x["do"], b, h), scale)
            for t in range(3):
                worst[t] = max(worst[t], maxerr(got[t][b, h], ref[t]))
    assert max(worst) <= tol, worst
    T = sp.kernel_tile(dtype, D)
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, layout)
    st = stats.cpu().numpy()
    assert np.array_equal(st[0], B * H * full) and np.array_equal(st[1], B * H * part)
    return worst


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 1, 256, 64, 4), (1, 2, 4 * 37, 32, 4), (2, 1, 96, 128, 8),
                                       (1, 1, 16, 64, 16),
                                       (1, 1, 4 * 45, 8, 4),    # D = 8: one element of a row per thread
                                       (1, 2, 144, 96, 3)])     # D = 96: the run-time head width, 12 per thread
def test_bwd_fp32(B, H, S, D, N, layout):
    x, grads, stats = _run(B, H, S, D, N, layout, torch.float32)
    _check(x, grads, stats, B, H, S, D, N, layout, torch.float32)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 2, 1200, 128, 4), (1, 1, 1028, 128, 4), (2, 1, 512, 128, 4),
                                       (1, 1, 256, 128, 4), (1, 1, 384, 128, 1), (1, 1, 48, 128, 16)])
def test_bwd_bf16_small(B, H, S, D, N, layout):
    x, grads, stats = _run(B, H, S, D, N, layout, torch.bfloat16, seed=1)
    _check(x, grads, stats, B, H, S, D, N, layout, torch.bfloat16)


@pytest.mark.parametrize("B,H,S,D,N", [(1, 1, 256, 64, 4), (1, 2, 128, 32, 4), (2, 1, 256, 128, 8),
                                       (1, 1, 512, 64, 16)])
def test_bwd_fp32_zigzag(B, H, S, D, N):
    x, grads, stats = _run(B, H, S, D, N, sp.ZIGZAG, torch.float32)
    _check(x, grads, stats, B, H, S, D, N, sp.ZIGZAG, torch.float32)


@pytest.mark.parametrize("B,H,S,D,N", [(1, 2, 1024, 128, 4), (2, 1, 2048, 128, 4), (1, 1, 512, 128, 1),
                                       (1, 1, 4096, 128, 16)])
def test_bwd_bf16_zigzag(B, H, S, D, N):
    x, grads, stats = _run(B, H, S, D, N, sp.ZIGZAG, torch.bfloat16, seed=1)
    _check(x, grads, stats, B, H, S, D, N, sp.ZIGZAG, torch.bfloat16)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 2, 2048, 64, 4), (2, 1, 2048, 64, 8)])
def test_bwd_bf16_head_dim_64(B, H, S, D, N, layout):
    x, grads, stats = _run(B, H, S, D, N, layout, torch.bfloat16, seed=5)
    _check(x, grads, stats, B, H, S, D, N, layout, torch.bfloat16)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
def test_bwd_bf16_head_dim_64_ragged(layout):
    """D = 64 with a ragged stripe tail (L = 300)."""
    B, H, S, D, N = 1, 2, 1200, 64, 4
    x, grads, stats = _run(B, H, S, D, N, layout, torch.bfloat16, seed=6)
    _check(x, grads, stats, B, H, S, D, N, layout, torch.bfloat16)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
def test_bwd_bf16_short_sequence_full(layout):
    """Short-sequence workload B=1, H=8, S=8192, D=128, N=8: every row."""
    B, H, S, D, N = 1, 8, 8192, 128, 8
    x, grads, stats = _run(B, H, S, D, N, layout, torch.bfloat16)
    print("max errors dq dk dv:", _check(x, grads, stats, B, H, S, D, N, layout, torch.bfloat16))


def test_bwd_invariants_on_device():
    """sum_t dV_t = sum_p dO_p and sum_t dK_t = 0 per head and column, on the
    full GPU tensors, under the bf16 error model of grad_sum_errors."""
    B, H, S, D, N = 1, 4, 4096, 128, 8
    x, (dq, dk, dv), _ = _run(B, H, S, D, N, sp.STRIPED, torch.bfloat16, seed=7)
    pos = torch.as_tensor(oracle.layout_positions(S, N, sp.STRIPED), device=DEV)
    inv = grad_sum_errors(dv, dk, x["do"].to(DEV), x["q"].to(DEV), pos)
    print("gradient invariants", inv)
    assert inv["dv"][2] <= 1.0 and inv["dk"][2] <= 1.0, inv


def test_bwd_workspace_contents_ignored():
    """Garbage in the caller's workspace does not change the result.  dQ is
    summed with fp32 atomics, so two runs agree up to summation order (a few
    fp32 ulps before the bf16 rounding), not bit for bit; dK and dV are
    accumulated in a fixed order and agree exactly."""
    B, H, S, D, N = 1, 1, 1024, 128, 4
    x = inputs(B, H, S, D, torch.bfloat16, seed=8)
    q, k, v, do = (to_layout(x[n], N, sp.STRIPED, DEV) for n in ("q", "k", "v", "do"))
    o, lse = sp.striped_attn_fwd(q, k, v, N)
    ws = sp.new_workspace(B, H, S, D, N, torch.bfloat16, DEV)
    ws.fill_(0x7f)
    g1 = sp.striped_attn_bwd(q, k, v, o, lse, do, N, workspace=ws)
    ws.fill_(0x11)
    g2 = sp.striped_attn_bwd(q, k, v, o, lse, do, N, workspace=ws)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert maxerr(g1[0].float().cpu(), g2[0].float().cpu()) <= 1e-2
