"""The ring protocol on the CPU (research.elamur.ai summary page, §Summary:
key/value blocks circulate between devices): world_size 2 and 4 gloo
processes, each holding one stripe (or contiguous / zig-zag block) of the
sequence as its own tensors, pass K/V blocks to rank + 1 every round and,
in the backward, the blocks' gradient sums with them.  The per-round
arithmetic is the oracle's (fp64, tests/_ring_util.py), so what is checked
is the protocol: in round r rank d holds block (d - r) mod N, the merged
round partials equal full causal attention, and every block's dK / dV sums
visit all ranks and come back to their owner complete."""
import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import attention_inputs
from tests._ring_util import OracleRoundCompute, spawn_ranks

STRIPED, CONTIGUOUS, ZIGZAG = 0, 1, 2


def _ring_rank(rank, world, layout, S, D, H):
    from sequence_parallelism_striped_gb300.ring import StripedRing, TorchDistTransport

    x = attention_inputs(1, H, S, D, torch.float32, seed=40)
    full = {n: x[n].double() for n in x}
    scale = 1.0 / D ** 0.5
    pos = oracle.layout_positions(S, world, layout)
    L = S // world
    mine = pos[rank * L:(rank + 1) * L]
    blk = {n: full[n][:, :, mine].contiguous() for n in full}
    comp = OracleRoundCompute(world, layout, S, scale, pos)
    ring = StripedRing(TorchDistTransport(), comp)
    k_before = blk["k"].clone()
    o, lse = ring.forward(blk["q"], blk["k"], blk["v"])
    dq, dk, dv = ring.backward(blk["q"], blk["k"], blk["v"], o, lse, blk["do"])
    err = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    for h in range(H):
        args = [full[n][0, h].numpy() for n in ("q", "k", "v", "do")]
        o_r, l_r = oracle.attn_fwd(args[0], args[1], args[2], scale)
        gq, gk, gv = oracle.attn_bwd(*args, scale)
        for name, got, ref in (("o", o, o_r), ("lse", lse, l_r), ("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
            err[name] = max(err[name], float(np.abs(got[0, h].numpy() - ref[mine]).max()))
    order = [(kind, d, e) for kind, d, e in comp.visits]
    want = [(kind, rank, (rank - r) % world) for kind in ("fwd", "bwd") for r in range(world)]
    return {"err": err, "order_ok": order == want, "k_untouched": bool(torch.equal(k_before, blk["k"]))}


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("layout", [STRIPED, CONTIGUOUS, ZIGZAG])
def test_ring_protocol_on_gloo(world, layout):
    S, D, H = 16 * world, 8, 2
    res = spawn_ranks(world, _ring_rank, (layout, S, D, H))
    for r in range(world):
        assert not isinstance(res[r], str), res[r]
        assert res[r]["order_ok"] and res[r]["k_untouched"], res[r]
        assert max(res[r]["err"].values()) < 1e-10, res[r]["err"]
