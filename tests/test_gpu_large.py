"""Full-size parity on the benchmark workloads (the launch configuration the
bench times): 4096 seed-sampled (b, h, position) query rows for O, LSE and
dQ against the fp64 oracle; dK and dV for key positions sampled from the
tail of one seed-chosen head (the oracle needs LSE and the Jacobian sums of
every query at or after a key, which is cheap only near the end); the
per-round tile counters against the oracle's closed forms; and the gradient
invariants sum_t dV_t = sum_p dO_p and sum_t dK_t = 0 on every head."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs, sample_head, sample_rows, sample_tail_keys

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda")

WORKLOADS = {
    "mid": (1, 24, 65536, 128, 8),
    "long": (1, 32, 262144, 128, 8),
    "vlong": (1, 16, 786432, 128, 16),
}


def _row_of_position(p, S, N):
    """Striped row holding position p (test-side inverse of the oracle map)."""
    L = S // N
    return (p % N) * L + p // N


@pytest.mark.parametrize("name", ["mid", "long", "vlong"])
def test_full_size_sampled_parity(name):
    B, H, S, D, N = WORKLOADS[name]
    scale = 1.0 / D ** 0.5
    x = attention_inputs(B, H, S, D, torch.bfloat16, seed=0)
    # the product path: permute on the GPU, forward, backward
    q, k, v, do = (sp.striped_permute(x[n].to(DEV), N) for n in ("q", "k", "v", "do"))
    stats = sp.new_tile_stats(N, DEV)
    o, lse = sp.striped_attn_fwd(q, k, v, N, sp.STRIPED, tile_stats=stats)
    dq, dk, dv = sp.striped_attn_bwd(q, k, v, o, lse, do, N, sp.STRIPED)
    torch.cuda.synchronize()
    assert sp.check_error() == 0

    # tile counters: B*H x the oracle's closed-form per-round table
    full, part = oracle.tile_counts_closed(S, N, 128, sp.STRIPED)
    st = stats.cpu().numpy()
    assert np.array_equal(st[0], B * H * full) and np.array_equal(st[1], B * H * part)

    # invariants on every head (fp64 sums of the GPU tensors)
    sdv = dv.double().sum(2)
    sdo = x["do"].to(DEV).double().sum(2)
    bound_v = np.sqrt(S) * 2.0 ** -9 * float(dv.abs().max()) + 2e-2
    assert float((sdv - sdo).abs().max()) <= bound_v
    bound_k = np.sqrt(S) * 2.0 ** -9 * float(dk.abs().max()) + 2e-2
    assert float(dk.double().sum(2).abs().max()) <= bound_k

    # 4096 sampled query rows: O, LSE, dQ
    rows = sample_rows(4096, B, H, S, seed=0).numpy()
    srow = _row_of_position(rows[:, 2], S, N)
    idx = torch.as_tensor(srow, device=DEV)
    bidx = torch.as_tensor(rows[:, 0], device=DEV)
    hidx = torch.as_tensor(rows[:, 1], device=DEV)
    o_s = o[bidx, hidx, idx].double().cpu().numpy()
    lse_s = lse[bidx, hidx, idx].double().cpu().numpy()
    dq_s = dq[bidx, hidx, idx].double().cpu().numpy()
    worst = {"o": 0.0, "lse": 0.0, "dq": 0.0}
    for (b, h) in sorted({(int(r[0]), int(r[1])) for r in rows}):
        sel = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
        pos = rows[sel, 2]
        args = [x[n][b, h].double().numpy() for n in ("q", "k", "v", "do")]
        o_ref, lse_ref = oracle.attn_fwd(args[0], args[1], args[2], scale, rows=pos)
        _, _, dq_ref = oracle.bwd_rows(*args, scale, rows=pos)
        worst["o"] = max(worst["o"], float(np.abs(o_s[sel] - o_ref).max()))
        worst["lse"] = max(worst["lse"], float(np.abs(lse_s[sel] - lse_ref).max()))
        worst["dq"] = max(worst["dq"], float(np.abs(dq_s[sel] - dq_ref).max()))
    print(name, "sampled max errors", worst)
    assert worst["o"] <= 2e-2 and worst["dq"] <= 2e-2 and worst["lse"] <= 1e-3, worst

    # dK, dV for 256 key positions from the last 1024 positions of one head
    b, h = sample_head(B, H, seed=0)
    keys = sample_tail_keys(256, S, 1024, seed=0).numpy()
    kidx = torch.as_tensor(_row_of_position(keys, S, N), device=DEV)
    dk_s = dk[b, h, kidx].double().cpu().numpy()
    dv_s = dv[b, h, kidx].double().cpu().numpy()
    args = [x[n][b, h].double().numpy() for n in ("q", "k", "v", "do")]
    dk_ref, dv_ref = oracle.bwd_keys(*args, scale, keys)
    ek, ev = float(np.abs(dk_s - dk_ref).max()), float(np.abs(dv_s - dv_ref).max())
    print(name, "tail-key max errors dk dv", ek, ev)
    assert ek <= 2e-2 and ev <= 2e-2
