"""The ring itself: N processes, one stripe each, key/value blocks passed
around the ring (research.elamur.ai summary page, §Summary: key/value blocks
circulate between devices while compute overlaps communication; pith.science
paper page, abstract).

Each process (rank d of N) holds its own stripe of the sequence -- rows of
positions p = i*N + d in the striped placement (or its contiguous / zig-zag
block) -- as contiguous [B, H, L, D] tensors.  In ring round r it holds the
key/value block of stripe e = (d - r) mod N and:

* forward: sends that block on to rank d + 1 and receives the next one from
  rank d - 1 while its round runs (``ring_round_fwd``: the round's partial
  result merged into the running (O, LSE) accumulator);
* backward: the block's fp32 dK / dV sums travel with it; rank d adds its
  round's share (``ring_round_bwd``) and passes block and sums on, so after
  N rounds every block's sums have visited all N ranks and come back to
  their owner.  dQ stays on its rank.

The transport moves tensors between ranks; ``TorchDistTransport`` uses
``torch.distributed`` point-to-point operations (NCCL moves device tensors
directly; gloo stages them through host memory).  The per-round arithmetic
is a ``RoundCompute``: ``CudaRoundCompute`` calls the library's kernels.
No arithmetic of the method happens in this module.
"""
from __future__ import annotations

import torch

from . import STRIPED
from . import ring_bwd_finish, ring_bwd_prepare, ring_bwd_workspace, ring_round_bwd, ring_round_fwd_block


class _Handle:
    def __init__(self, reqs, post=None):
        self.reqs = reqs
        self.post = post

    def wait(self):
        for r in self.reqs:
            r.wait()
        if self.post is not None:
            self.post()


class TorchDistTransport:
    """One ring step over a torch.distributed process group: every rank
    sends tensors to rank + 1 and receives the same shapes from rank - 1,
    asynchronously.  With NCCL the device tensors move directly; with gloo
    they are staged through host memory (gloo moves host tensors only)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.backend = dist.get_backend(group)

    def _peer(self, r):
        return self.dist.get_global_rank(self.group, r) if self.group is not None else r

    def shift(self, send, recv) -> _Handle:
        dist = self.dist
        nxt = self._peer((self.rank + 1) % self.world)
        prv = self._peer((self.rank - 1) % self.world)
        if self.backend == "nccl":
            ops = [dist.P2POp(dist.isend, t, nxt, self.group) for t in send]
            ops += [dist.P2POp(dist.irecv, t, prv, self.group) for t in recv]
            return _Handle(dist.batch_isend_irecv(ops))

        def host(t):  # bytes of t on the host (gloo: any dtype as raw 16/32-bit words)
            h = t.detach().to("cpu", copy=True)
            return h.view(torch.int16) if h.dtype == torch.bfloat16 else h

        hs = [host(t) for t in send]
        hr = [torch.empty(t.shape, dtype=torch.int16 if t.dtype == torch.bfloat16 else t.dtype) for t in recv]
        reqs = [dist.isend(h, nxt, group=self.group) for h in hs]
        reqs += [dist.irecv(h, prv, group=self.group) for h in hr]

        def post():
            for t, h in zip(recv, hr):
                t.copy_(h.view(t.dtype) if t.dtype == torch.bfloat16 else h, non_blocking=False)

        return _Handle(reqs, post)


class CudaRoundCompute:
    """The per-round work of one rank on its GPU (bf16, the library's
    kernels)."""

    def __init__(self, N: int, layout: int = STRIPED, scale: float | None = None):
        self.N = N
        self.layout = layout
        self.scale = scale

    def _scale(self, D):
        return self.scale if self.scale is not None else 1.0 / D ** 0.5

    # forward
    def fwd_begin(self, q_d):
        B, H, L, D = q_d.shape
        o_acc = torch.empty(B, H, L, D, dtype=torch.float32, device=q_d.device)
        lse_acc = torch.empty(B, H, L, dtype=torch.float32, device=q_d.device)
        return {"o_acc": o_acc, "lse": lse_acc, "o": torch.empty_like(q_d)}

    def fwd_round(self, ctx, q_d, k_e, v_e, d, e, first, last, tile_stats=None):
        ring_round_fwd_block(q_d, k_e, v_e, ctx["o_acc"], ctx["lse"], d, e, self.N, self.layout,
                             self._scale(q_d.shape[-1]), first_round=first, o_out=ctx["o"] if last else None,
                             tile_stats=tile_stats)

    def fwd_end(self, ctx):
        return ctx["o"], ctx["lse"]

    # backward
    def bwd_begin(self, q_d, o_d, lse_d, dO_d):
        ws = ring_bwd_workspace(q_d)
        dq_acc = torch.empty(q_d.shape, dtype=torch.float32, device=q_d.device)
        ring_bwd_prepare(o_d, lse_d, dO_d, ws, dq_acc)
        return {"ws": ws, "dq_acc": dq_acc}

    def new_grad_sums(self, k_d):
        return [torch.empty(k_d.shape, dtype=torch.float32, device=k_d.device) for _ in range(2)]

    def bwd_round(self, ctx, q_d, k_e, v_e, dO_d, dk_acc, dv_acc, d, e, first, tile_stats=None):
        ring_round_bwd(q_d, k_e, v_e, dO_d, ctx["ws"], ctx["dq_acc"], dk_acc, dv_acc, d, e, self.N, self.layout,
                       self._scale(q_d.shape[-1]), first_round=first, tile_stats=tile_stats)

    def bwd_end(self, ctx, dk_acc, dv_acc):
        D = dk_acc.shape[-1]
        return (ring_bwd_finish(ctx["dq_acc"], self._scale(D)), ring_bwd_finish(dk_acc, 1.0),
                ring_bwd_finish(dv_acc, 1.0))


class StripedRing:
    """Rank d's side of the ring (rank and N from the transport)."""

    def __init__(self, transport, compute):
        self.t = transport
        self.c = compute
        self.d = transport.rank
        self.N = transport.world

    def forward(self, q_d, k_d, v_d, tile_stats=None):
        """(O_d, LSE_d) of this rank's query block over all N rounds."""
        ctx = self.c.fwd_begin(q_d)
        bufs = [[torch.empty_like(k_d), torch.empty_like(v_d)] for _ in range(2)]  # the caller's stay untouched
        cur = [k_d, v_d]
        for r in range(self.N):
            e = (self.d - r) % self.N
            nxt = bufs[r % 2]
            h = self.t.shift(cur, nxt) if r + 1 < self.N else None  # next block arrives during the round
            self.c.fwd_round(ctx, q_d, cur[0], cur[1], self.d, e, r == 0, r + 1 == self.N, tile_stats)
            if h is not None:
                h.wait()
                cur = nxt
        return self.c.fwd_end(ctx)

    def backward(self, q_d, k_d, v_d, o_d, lse_d, dO_d, tile_stats=None):
        """(dQ_d, dK_d, dV_d) of this rank's blocks."""
        ctx = self.c.bwd_begin(q_d, o_d, lse_d, dO_d)
        bufs = [[torch.empty_like(k_d), torch.empty_like(v_d)] for _ in range(2)]
        cur = [k_d, v_d]
        g_cur = self.c.new_grad_sums(k_d)
        g_nxt = self.c.new_grad_sums(k_d)
        for r in range(self.N):
            e = (self.d - r) % self.N
            nxt = bufs[r % 2]
            hk = self.t.shift(cur, nxt) if r + 1 < self.N else None  # the next K/V during the round
            self.c.bwd_round(ctx, q_d, cur[0], cur[1], dO_d, g_cur[0], g_cur[1], self.d, e, r == 0, tile_stats)
            # the block's sums follow it; after the last round they reach its owner
            hg = self.t.shift(g_cur, g_nxt)
            if hk is not None:
                hk.wait()
                cur = nxt
            hg.wait()
            g_cur, g_nxt = g_nxt, g_cur
        return self.c.bwd_end(ctx, g_cur[0], g_cur[1])
