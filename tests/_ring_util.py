"""Shared pieces of the ring-protocol tests: the oracle-backed per-round
compute (fp64, host) and the per-rank process driver.  Test code only."""
import os
import socket
import traceback

import numpy as np
import torch

import oracle


def free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class OracleRoundCompute:
    """The per-round arithmetic of one rank, in fp64 on the host, by the
    oracle: a round's forward partial is the oracle's attention restricted
    to the round's key block (merged in ring order by the log-sum-exp rule),
    a round's gradient share is oracle.bwd_block.  Blocks are CPU float64
    tensors [B, H, L, D]; `pos` maps a layout row to its position."""

    def __init__(self, N, layout, S, scale, pos):
        self.N, self.layout, self.S, self.scale, self.pos = N, layout, S, scale, pos
        self.L = S // N
        self.visits = []  # (direction, d, e) in the order the rounds ran

    def _rows(self, x):
        return self.pos[x * self.L:(x + 1) * self.L]

    def fwd_begin(self, q_d):
        B, H, L, D = q_d.shape
        return {"o": np.zeros((B, H, L, D)), "lse": np.full((B, H, L), -np.inf)}

    def fwd_round(self, ctx, q_d, k_e, v_e, d, e, first, last, tile_stats=None):
        self.visits.append(("fwd", d, e))
        qp, kp = self._rows(d), self._rows(e)
        keys = np.zeros(self.S, dtype=bool)
        keys[kp] = True
        B, H, L, D = q_d.shape
        for b in range(B):
            for h in range(H):
                qf, kf, vf = (np.zeros((self.S, D)) for _ in range(3))
                qf[qp] = q_d[b, h].numpy()
                kf[kp] = k_e[b, h].numpy()
                vf[kp] = v_e[b, h].numpy()
                o_r, l_r = oracle.attn_fwd(qf, kf, vf, self.scale, rows=qp, key_in_set=keys)
                if first:
                    ctx["o"][b, h], ctx["lse"][b, h] = o_r, l_r
                else:
                    ctx["o"][b, h], ctx["lse"][b, h] = oracle.merge_rounds(ctx["o"][b, h], ctx["lse"][b, h], o_r, l_r)

    def fwd_end(self, ctx):
        return torch.from_numpy(ctx["o"]), torch.from_numpy(ctx["lse"])

    def bwd_begin(self, q_d, o_d, lse_d, dO_d):
        J = (dO_d.numpy() * o_d.numpy()).sum(-1)  # J_p = <dO_p, O_p>
        return {"dq": np.zeros(q_d.shape), "J": J, "lse": lse_d.numpy()}

    def new_grad_sums(self, k_d):
        return [torch.zeros(k_d.shape, dtype=torch.float64) for _ in range(2)]

    def bwd_round(self, ctx, q_d, k_e, v_e, dO_d, dk_acc, dv_acc, d, e, first, tile_stats=None):
        self.visits.append(("bwd", d, e))
        qp, kp = self._rows(d), self._rows(e)
        B, H = q_d.shape[:2]
        for b in range(B):
            for h in range(H):
                gq, gk, gv = oracle.bwd_block(q_d[b, h].numpy(), dO_d[b, h].numpy(), qp, ctx["lse"][b, h],
                                              ctx["J"][b, h], k_e[b, h].numpy(), v_e[b, h].numpy(), kp, self.scale)
                ctx["dq"][b, h] += gq
                if first:
                    dk_acc[b, h] = torch.from_numpy(gk)
                    dv_acc[b, h] = torch.from_numpy(gv)
                else:
                    dk_acc[b, h] += torch.from_numpy(gk)
                    dv_acc[b, h] += torch.from_numpy(gv)

    def bwd_end(self, ctx, dk_acc, dv_acc):
        return torch.from_numpy(ctx["dq"]), dk_acc.clone(), dv_acc.clone()


def run_rank(rank, world, port, fn, args, queue):
    """Process body: join the gloo group on 127.0.0.1, run fn(rank, world,
    *args), report (rank, result or the error text)."""
    import torch.distributed as dist

    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        try:
            queue.put((rank, fn(rank, world, *args)))
        finally:
            dist.destroy_process_group()
    except Exception:  # the parent reports it
        queue.put((rank, "error:\n" + traceback.format_exc()))


def spawn_ranks(world, fn, args, timeout=600):
    """Run fn on `world` spawned processes; return {rank: result}."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=run_rank, args=(r, world, port, fn, args, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(world):
            r, res = q.get(timeout=timeout)
            out[r] = res
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    return out
