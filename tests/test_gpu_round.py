"""ring_round_fwd: N per-round calls per virtual device, merged by the LSE
rule, reproduce the oracle; per-round tile counts equal the batched ones."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from tests._util import TOL, head64, inputs, maxerr, to_layout, to_positions

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("dtype,B,H,S,D,N", [(torch.float32, 1, 1, 256, 64, 4),
                                             (torch.bfloat16, 1, 2, 1200, 128, 4),
                                             (torch.bfloat16, 1, 1, 1028, 128, 4),
                                             (torch.bfloat16, 1, 4, 8192, 128, 8),
                                             (torch.bfloat16, 1, 2, 1200, 64, 4)])
@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
def test_rounds_merge_to_full_attention(dtype, B, H, S, D, N, layout):
    _rounds_merge(dtype, B, H, S, D, N, layout)


@pytest.mark.parametrize("dtype,B,H,S,D,N", [(torch.float32, 1, 1, 256, 64, 4),
                                             (torch.bfloat16, 1, 2, 2048, 128, 4),
                                             (torch.bfloat16, 1, 4, 8192, 128, 8)])
def test_zigzag_rounds_merge_to_full_attention(dtype, B, H, S, D, N):
    _rounds_merge(dtype, B, H, S, D, N, sp.ZIGZAG)


def _rounds_merge(dtype, B, H, S, D, N, layout):
    x = inputs(B, H, S, D, dtype, seed=2, with_do=False)
    q, k, v = (to_layout(x[n], N, layout, DEV) for n in ("q", "k", "v"))
    o_acc = torch.empty(B, H, S, D, dtype=torch.float32, device=DEV)
    lse_acc = torch.empty(B, H, S, dtype=torch.float32, device=DEV)
    o_out = torch.empty_like(q)
    stats = sp.new_tile_stats(N, DEV)
    for d in range(N):
        for r in range(N):
            e = (d - r) % N
            sp.ring_round_fwd(q, k, v, o_acc, lse_acc, d, e, N, layout, first_round=(r == 0),
                              o_out=o_out if r == N - 1 else None, tile_stats=stats)
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    scale = 1.0 / D ** 0.5
    o_pos = to_positions(o_acc, N, layout)
    lse_pos = to_positions(lse_acc[..., None], N, layout)[..., 0]
    tol = TOL[dtype]
    for b in range(B):
        for h in range(H):
            o_ref, lse_ref = oracle.attn_fwd(head64(x["q"], b, h), head64(x["k"], b, h),
                                             head64(x["v"], b, h), scale)
            assert maxerr(o_pos[b, h], o_ref) <= tol["o"]
            assert maxerr(lse_pos[b, h], lse_ref) <= tol["lse"]
    # the dtype copy of the merged O is the rounded accumulator
    assert torch.equal(o_out, o_acc.to(dtype))
    T = sp.kernel_tile(dtype, D)
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, layout)
    st = stats.cpu().numpy()
    assert np.array_equal(st[0], B * H * full) and np.array_equal(st[1], B * H * part)


def test_single_round_partial_matches_oracle_keyset():
    """One round's partial result (first_round=1) is attention over exactly
    the key stripe e (rows with no kept key: O = 0, LSE = -inf)."""
    B, H, S, D, N = 1, 1, 1024, 128, 4
    L = S // N
    x = inputs(B, H, S, D, torch.bfloat16, seed=6, with_do=False)
    q, k, v = (to_layout(x[n], N, sp.STRIPED, DEV) for n in ("q", "k", "v"))
    scale = 1.0 / D ** 0.5
    pos = oracle.stripe_positions(S, N)
    for d, e in [(0, 3), (2, 1), (1, 1)]:
        o_acc = torch.zeros(B, H, S, D, dtype=torch.float32, device=DEV)
        lse_acc = torch.zeros(B, H, S, dtype=torch.float32, device=DEV)
        sp.ring_round_fwd(q, k, v, o_acc, lse_acc, d, e, N, sp.STRIPED, first_round=True)
        torch.cuda.synchronize()
        keyset = np.zeros(S, dtype=bool)
        keyset[pos[e * L:(e + 1) * L]] = True
        rows = pos[d * L:(d + 1) * L]
        o_ref, lse_ref = oracle.attn_fwd(head64(x["q"], 0, 0), head64(x["k"], 0, 0), head64(x["v"], 0, 0),
                                         scale, rows=rows, key_in_set=keyset)
        got_o = o_acc[0, 0, d * L:(d + 1) * L].cpu().numpy()
        got_l = lse_acc[0, 0, d * L:(d + 1) * L].cpu().numpy()
        assert maxerr(got_o, o_ref) <= 2e-2
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(got_l), fin)
        assert maxerr(got_l[fin], lse_ref[fin]) <= 1e-3


def test_rounds_captured_in_a_cuda_graph():
    """The per-round path is launch-bound at short sequences; its N x N
    ring_round_fwd launches can be captured in one CUDA graph (the library
    launches only on the caller's stream and its one-time set-up runs on the
    first, eager call).  Replaying the graph reproduces the eager result
    exactly, including on new inputs copied into the captured buffers."""
    B, H, S, D, N = 1, 4, 8192, 128, 8
    x = inputs(B, H, S, D, torch.bfloat16, seed=9, with_do=False)
    q, k, v = (to_layout(x[n], N, sp.STRIPED, DEV) for n in ("q", "k", "v"))
    o_acc = torch.empty(B, H, S, D, dtype=torch.float32, device=DEV)
    lse_acc = torch.empty(B, H, S, dtype=torch.float32, device=DEV)

    def rounds():
        for r in range(N):
            for d in range(N):
                sp.ring_round_fwd(q, k, v, o_acc, lse_acc, d, (d - r) % N, N, sp.STRIPED, first_round=(r == 0))

    rounds()  # eager: one-time set-up, reference result
    torch.cuda.synchronize()
    o_ref, l_ref = o_acc.clone(), lse_acc.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            rounds()
    torch.cuda.current_stream().wait_stream(s)
    o_acc.zero_()
    lse_acc.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    assert torch.equal(o_acc, o_ref) and torch.equal(lse_acc, l_ref)
    # new inputs through the same captured buffers
    y = inputs(B, H, S, D, torch.bfloat16, seed=10, with_do=False)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        t.copy_(to_layout(y[n], N, sp.STRIPED, DEV))
    graph.replay()
    rounds_out = (o_acc.clone(), lse_acc.clone())
    rounds()
    torch.cuda.synchronize()
    assert torch.equal(rounds_out[0], o_acc) and torch.equal(rounds_out[1], lse_acc)
