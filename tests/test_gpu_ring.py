"""The ring's per-round kernels on the GPU, and the ring itself with two
processes (research.elamur.ai summary page, §Summary: key/value blocks
circulate; each device accumulates the work of the block it holds).

1. One process, every device's blocks as their own tensors: N x N rounds of
   ring_round_fwd / ring_round_bwd in ring order (the gradient sums of block
   e start on device e and are added to by every device after it) against
   the fp64 oracle, with the per-round tile counters summed over devices
   equal to the oracle's table.
2. Two processes sharing this GPU, joined by gloo (blocks staged through
   host memory), each the rank of one stripe: StripedRing forward and
   backward against the oracle, tile counters gathered from both ranks.
   The ranks' kernels never wait on each other: every exchange is on the
   host, between launches."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs
from tests._ring_util import spawn_ranks
from tests._util import TOL

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _oracle_all(x, H, scale):
    out = []
    for h in range(H):
        args = [x[n][0, h].double().numpy() for n in ("q", "k", "v", "do")]
        o, l = oracle.attn_fwd(args[0], args[1], args[2], scale)
        gq, gk, gv = oracle.attn_bwd(*args, scale)
        out.append((o, l, gq, gk, gv))
    return out


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
@pytest.mark.parametrize("S,D,N", [(2048, 128, 4), (2048, 64, 4), (1200, 128, 4)])
def test_round_kernels_in_ring_order_match_oracle(layout, S, D, N):
    if layout == sp.ZIGZAG and (S // (2 * N)) % 128:
        pytest.skip("zig-zag attention needs whole 128-row chunks")
    H = 2
    L = S // N
    x = attention_inputs(1, H, S, D, torch.bfloat16, seed=44)
    scale = 1.0 / D ** 0.5
    pos = oracle.layout_positions(S, N, layout)
    blk = {n: [x[n][:, :, pos[d * L:(d + 1) * L]].contiguous().to(DEV) for d in range(N)] for n in x}
    fst, bst = sp.new_tile_stats(N, DEV), sp.new_tile_stats(N, DEV)
    o_acc = [torch.empty(1, H, L, D, dtype=torch.float32, device=DEV) for _ in range(N)]
    lse = [torch.empty(1, H, L, dtype=torch.float32, device=DEV) for _ in range(N)]
    o = [torch.empty(1, H, L, D, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    for r in range(N):
        for d in range(N):
            e = (d - r) % N
            sp.ring_round_fwd_block(blk["q"][d], blk["k"][e], blk["v"][e], o_acc[d], lse[d], d, e, N, layout,
                                    first_round=(r == 0), o_out=o[d] if r == N - 1 else None, tile_stats=fst)
    ws = [sp.ring_bwd_workspace(blk["q"][d]) for d in range(N)]
    dq_acc = [torch.empty(1, H, L, D, dtype=torch.float32, device=DEV) for _ in range(N)]
    for d in range(N):
        sp.ring_bwd_prepare(o[d], lse[d], blk["do"][d], ws[d], dq_acc[d])
    dk_acc = [torch.full((1, H, L, D), 7.0, device=DEV) for _ in range(N)]  # garbage: round 0 overwrites
    dv_acc = [torch.full((1, H, L, D), 7.0, device=DEV) for _ in range(N)]
    for r in range(N):
        for d in range(N):
            e = (d - r) % N
            sp.ring_round_bwd(blk["q"][d], blk["k"][e], blk["v"][e], blk["do"][d], ws[d], dq_acc[d], dk_acc[e],
                              dv_acc[e], d, e, N, layout, first_round=(r == 0), tile_stats=bst)
    dq = [sp.ring_bwd_finish(dq_acc[d], scale) for d in range(N)]
    dk = [sp.ring_bwd_finish(dk_acc[d], 1.0) for d in range(N)]
    dv = [sp.ring_bwd_finish(dv_acc[d], 1.0) for d in range(N)]
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    tol = TOL[torch.bfloat16]
    ref = _oracle_all(x, H, scale)
    worst = dict.fromkeys(("o", "lse", "dq", "dk", "dv"), 0.0)
    for d in range(N):
        rows = pos[d * L:(d + 1) * L]
        for h in range(H):
            o_r, l_r, gq, gk, gv = ref[h]
            for name, got, want in (("o", o[d], o_r), ("lse", lse[d], l_r), ("dq", dq[d], gq), ("dk", dk[d], gk),
                                    ("dv", dv[d], gv)):
                worst[name] = max(worst[name], float(np.abs(got[0, h].double().cpu().numpy() - want[rows]).max()))
    print("ring-order rounds max errors", worst)
    assert worst["o"] <= tol["o"] and worst["lse"] <= tol["lse"]
    assert worst["dq"] <= tol["grad"] and worst["dk"] <= tol["grad"] and worst["dv"] <= tol["grad"]
    full, part = oracle.tile_counts_bruteforce(S, N, 128, 128, layout)
    for st in (fst, bst):
        c = st.cpu().numpy()
        assert np.array_equal(c[0], H * full) and np.array_equal(c[1], H * part)


def _gpu_rank(rank, world, layout, S, D, H):
    import torch.distributed as dist

    import sequence_parallelism_striped_gb300 as spr
    from sequence_parallelism_striped_gb300.ring import CudaRoundCompute, StripedRing, TorchDistTransport

    dev = torch.device("cuda", 0)  # both ranks share the one GPU of this test
    torch.cuda.set_device(dev)
    x = attention_inputs(1, H, S, D, torch.bfloat16, seed=45)
    pos = oracle.layout_positions(S, world, layout)
    L = S // world
    mine = pos[rank * L:(rank + 1) * L]
    blk = {n: x[n][:, :, mine].contiguous().to(dev) for n in x}
    ring = StripedRing(TorchDistTransport(), CudaRoundCompute(world, layout))
    fst, bst = spr.new_tile_stats(world, dev), spr.new_tile_stats(world, dev)
    o, lse = ring.forward(blk["q"], blk["k"], blk["v"], tile_stats=fst)
    dq, dk, dv = ring.backward(blk["q"], blk["k"], blk["v"], o, lse, blk["do"], tile_stats=bst)
    torch.cuda.synchronize()
    status = spr.check_error()
    stats = torch.stack([fst, bst]).cpu()
    dist.all_reduce(stats)  # every rank wrote only its own device column
    scale = 1.0 / D ** 0.5
    worst = dict.fromkeys(("o", "lse", "dq", "dk", "dv"), 0.0)
    for h in range(H):
        args = [x[n][0, h].double().numpy() for n in ("q", "k", "v", "do")]
        o_r, l_r = oracle.attn_fwd(args[0], args[1], args[2], scale)
        gq, gk, gv = oracle.attn_bwd(*args, scale)
        for name, got, want in (("o", o, o_r), ("lse", lse, l_r), ("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
            worst[name] = max(worst[name], float(np.abs(got[0, h].double().cpu().numpy() - want[mine]).max()))
    return {"status": status, "worst": worst, "stats": stats.numpy()}


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
def test_ring_two_processes_on_one_gpu(layout):
    world, S, D, H = 2, 2048, 128, 2
    res = spawn_ranks(world, _gpu_rank, (layout, S, D, H))
    full, part = oracle.tile_counts_bruteforce(S, world, 128, 128, layout)
    tol = TOL[torch.bfloat16]
    for r in range(world):
        assert not isinstance(res[r], str), res[r]
        print("rank", r, res[r]["worst"])
        assert res[r]["status"] == 0
        w = res[r]["worst"]
        assert w["o"] <= tol["o"] and w["lse"] <= tol["lse"]
        assert w["dq"] <= tol["grad"] and w["dk"] <= tol["grad"] and w["dv"] <= tol["grad"]
        for st in res[r]["stats"]:
            assert np.array_equal(st[0], H * full) and np.array_equal(st[1], H * part)
