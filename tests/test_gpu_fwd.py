"""Forward parity on the GPU against the fp64 CPU oracle (on the unpermuted
sequence), plus the per-round tile counters against the oracle's brute
force.  Striped results are mapped back to position order on the host."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from tests._util import TOL, head64, inputs, maxerr, to_layout, to_positions

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run_fwd(B, H, S, D, N, layout, dtype, seed=0):
    x = inputs(B, H, S, D, dtype, seed=seed, with_do=False)
    q, k, v = (to_layout(x[n], N, layout, DEV) for n in ("q", "k", "v"))
    stats = sp.new_tile_stats(N, DEV)
    o, lse = sp.striped_attn_fwd(q, k, v, N, layout, tile_stats=stats)
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    return x, o, lse, stats


def _check_fwd(x, o, lse, stats, B, H, S, D, N, layout, dtype, heads=None):
    scale = 1.0 / D ** 0.5
    o_pos = to_positions(o, N, layout)
    lse_pos = to_positions(lse[..., None], N, layout)[..., 0]
    tol = TOL[dtype]
    worst_o = worst_l = 0.0
    for b in range(B):
        for h in (range(H) if heads is None else heads):
            o_ref, lse_ref = oracle.attn_fwd(head64(x["q"], b, h), head64(x["k"], b, h),
                                             head64(x["v"], b, h), scale)
            worst_o = max(worst_o, maxerr(o_pos[b, h], o_ref))
            worst_l = max(worst_l, maxerr(lse_pos[b, h], lse_ref))
    assert worst_o <= tol["o"], worst_o
    assert worst_l <= tol["lse"], worst_l
    T = sp.kernel_tile(dtype, D)
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, layout)
    st = stats.cpu().numpy()
    assert np.array_equal(st[0], B * H * full) and np.array_equal(st[1], B * H * part)
    return worst_o, worst_l


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 1, 256, 64, 4), (1, 2, 4 * 37, 32, 4), (2, 1, 96, 128, 8),
                                       (1, 1, 64, 64, 1), (1, 1, 16, 64, 16),
                                       (1, 1, 4 * 45, 8, 4),    # D = 8: one element of a row per thread
                                       (1, 2, 144, 96, 3)])     # D = 96: the run-time head width, 12 per thread
def test_fwd_fp32(B, H, S, D, N, layout):
    x, o, lse, stats = _run_fwd(B, H, S, D, N, layout, torch.float32)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, layout, torch.float32)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 2, 1200, 128, 4),   # L=300: 128+128+44 rows
                                       (1, 1, 1028, 128, 4),   # L=257: last tile has one row
                                       (2, 1, 512, 128, 4),    # L=128: one full tile
                                       (1, 1, 256, 128, 4),    # L=64 < tile
                                       (1, 1, 384, 128, 1),    # N=1: plain causal attention
                                       (1, 1, 48, 128, 16)])   # L=3
def test_fwd_bf16_small(B, H, S, D, N, layout):
    x, o, lse, stats = _run_fwd(B, H, S, D, N, layout, torch.bfloat16, seed=1)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, layout, torch.bfloat16)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
def test_fwd_bf16_short_sequence_full(layout):
    """Short-sequence workload B=1, H=8, S=8192, D=128, N=8: every row."""
    B, H, S, D, N = 1, 8, 8192, 128, 8
    x, o, lse, stats = _run_fwd(B, H, S, D, N, layout, torch.bfloat16)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, layout, torch.bfloat16)


@pytest.mark.parametrize("B,H,S,D,N,pairs", [(1, 24, 8192, 128, 8, 2),   # 8 tiles a stripe, 4 stripe pairs
                                             (2, 24, 4096, 128, 2, 2),   # one stripe pair, 16 tiles a stripe
                                             (1, 24, 6144, 128, 6, 2),   # N = 6
                                             (1, 8, 8192, 128, 8, 1),    # too few tiles per SM for pairs
                                             (1, 2, 1536, 128, 3, 1),    # odd N
                                             (1, 24, 8192, 64, 8, 2),    # head dimension 64
                                             (2, 24, 4096, 64, 2, 2)])
def test_fwd_bf16_stripe_pairs(B, H, S, D, N, pairs):
    """Whole-tile stripes, an even N and enough work per multiprocessor: the
    forward runs the query tiles of stripes d and d + 1 in one CTA on one
    K/V stream (checked against the oracle on a few heads of each batch).
    `pairs` is the schedule on a 152-SM GB300; the balance rule is
    re-derived here for the device the test runs on."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    L = S // N
    nq = L // 128
    if N % 2 == 0 and L % 128 == 0:
        want = 2 if 2 * (2 * nq * N) * sms <= B * H * N * N * nq * (nq + 1) // 2 else 1
    else:
        want = 1
    if sms == 152:
        assert want == pairs
    assert sp.fwd_query_tiles_per_cta(B, H, S, D, N, sp.STRIPED) == want
    x, o, lse, stats = _run_fwd(B, H, S, D, N, sp.STRIPED, torch.bfloat16, seed=4)
    heads = sorted({0, H // 2, H - 1})
    _check_fwd(x, o, lse, stats, B, H, S, D, N, sp.STRIPED, torch.bfloat16, heads=heads)


@pytest.mark.parametrize("B,H,S,D,N", [(1, 1, 256, 64, 4), (1, 2, 128, 32, 4), (2, 1, 256, 128, 8),
                                       (1, 1, 64, 64, 1), (1, 1, 512, 64, 16)])
def test_fwd_fp32_zigzag(B, H, S, D, N):
    x, o, lse, stats = _run_fwd(B, H, S, D, N, sp.ZIGZAG, torch.float32)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, sp.ZIGZAG, torch.float32)


@pytest.mark.parametrize("B,H,S,D,N", [(1, 2, 1024, 128, 4),   # one tile per chunk
                                       (2, 1, 2048, 128, 4),   # two tiles per chunk
                                       (1, 1, 512, 128, 1),    # N=1: plain causal attention
                                       (1, 1, 4096, 128, 16)])
def test_fwd_bf16_zigzag(B, H, S, D, N):
    x, o, lse, stats = _run_fwd(B, H, S, D, N, sp.ZIGZAG, torch.bfloat16, seed=1)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, sp.ZIGZAG, torch.bfloat16)


def test_fwd_bf16_zigzag_short_sequence_full():
    """Short-sequence workload B=1, H=8, S=8192, D=128, N=8, zig-zag
    placement: every row, and the per-round counters (no partial tile after
    round 0)."""
    B, H, S, D, N = 1, 8, 8192, 128, 8
    x, o, lse, stats = _run_fwd(B, H, S, D, N, sp.ZIGZAG, torch.bfloat16)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, sp.ZIGZAG, torch.bfloat16)
    assert int(stats[1, 1:].sum()) == 0


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 2, 2048, 64, 4),    # head dimension 64: one 64-column box
                                       (2, 1, 2048, 64, 8)])
def test_fwd_bf16_head_dim_64(B, H, S, D, N, layout):
    x, o, lse, stats = _run_fwd(B, H, S, D, N, layout, torch.bfloat16, seed=5)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, layout, torch.bfloat16)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
def test_fwd_bf16_head_dim_64_ragged(layout):
    """D = 64 with a ragged stripe tail (L = 300)."""
    B, H, S, D, N = 1, 2, 1200, 64, 4
    x, o, lse, stats = _run_fwd(B, H, S, D, N, layout, torch.bfloat16, seed=6)
    _check_fwd(x, o, lse, stats, B, H, S, D, N, layout, torch.bfloat16)


def test_striped_equals_contiguous_after_unpermute():
    """Permutation equivariance on the GPU path itself: striped output mapped
    back to positions equals the contiguous-layout output."""
    B, H, S, D, N = 1, 2, 2048, 128, 8
    x = inputs(B, H, S, D, torch.bfloat16, seed=3, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o_c, lse_c = sp.striped_attn_fwd(q, k, v, N, sp.CONTIGUOUS)
    qs, ks, vs = (sp.striped_permute(t, N) for t in (q, k, v))
    o_s, lse_s = sp.striped_attn_fwd(qs, ks, vs, N, sp.STRIPED)
    o_back = sp.striped_unpermute(o_s, N)
    assert maxerr(o_back.float().cpu(), o_c.float().cpu()) <= 2e-2
    lse_back = to_positions(lse_s[..., None], N, sp.STRIPED)[..., 0]
    assert maxerr(lse_back, lse_c.cpu().numpy()) <= 1e-3


def test_first_position_attends_itself():
    """Position 0 keeps one key: O_0 = v_0 (to bf16 rounding)."""
    B, H, S, D, N = 1, 1, 1024, 128, 8
    x, o, lse, stats = _run_fwd(B, H, S, D, N, sp.STRIPED, torch.bfloat16, seed=4)
    assert maxerr(o[0, 0, 0].float().cpu(), x["v"][0, 0, 0].float()) <= 1e-2
