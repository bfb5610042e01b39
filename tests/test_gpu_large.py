"""Full-size parity on the benchmark workloads (the launch configuration the
bench times): 4096 seed-sampled (b, h, position) query rows for O, LSE and
dQ against the fp64 oracle; dK and dV for 4096 key positions drawn
uniformly over the whole sequence of one seed-chosen head (the oracle first
runs a full-head fp64 pass for the LSE and Jacobian sum of every query,
about 2 D S^2 flops: seconds at S = 65,536, minutes at 262,144), so the
early key tiles, which accumulate dK/dV over every later query tile of all
N stripes, are compared element by element; at S = 786,432 that pass would
take about an hour, so there the keys come from the last 1,024 positions;
the per-round tile counters against the oracle's closed forms; and the
gradient invariants sum_t dV_t = sum_p dO_p and sum_t dK_t = 0 on every
head and column, under an error bound that grows like sqrt(log S)."""
import time

import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs, sample_head, sample_keys, sample_rows, sample_tail_keys
from tests._util import grad_sum_errors

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
    t_rows = time.perf_counter()
    for (b, h) in sorted({(int(r[0]), int(r[1])) for r in rows}):
        sel = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
        pos = rows[sel, 2]
        args = [x[n][b, h].double().numpy() for n in ("q", "k", "v", "do")]
        o_ref, lse_ref = oracle.attn_fwd(args[0], args[1], args[2], scale, rows=pos)
        _, _, dq_ref = oracle.bwd_rows(*args, scale, rows=pos)
        worst["o"] = max(worst["o"], float(np.abs(o_s[sel] - o_ref).max()))
        worst["lse"] = max(worst["lse"], float(np.abs(lse_s[sel] - lse_ref).max()))
        worst["dq"] = max(worst["dq"], float(np.abs(dq_s[sel] - dq_ref).max()))
    t_rows = time.perf_counter() - t_rows
    print(name, "sampled max errors", worst, f"(oracle: 4096 query rows in {t_rows:.1f} s on "
          f"{oracle.default_threads()} threads)")
    assert worst["o"] <= 2e-2 and worst["dq"] <= 2e-2 and worst["lse"] <= 1e-3, worst

    # dK, dV of one seed-chosen head: 4096 keys uniform over [0, S) (the
    # oracle's full-head pass), or 256 of the last 1024 at the largest size
    b, h = sample_head(B, H, seed=0)
    if name == "vlong":
        keys = sample_tail_keys(256, S, 1024, seed=0).numpy()
        what = "256 tail keys"
    else:
        keys = sample_keys(4096, S, seed=0).numpy()
        assert keys.min() < S // 64 and keys.max() > S - S // 64
        what = "4096 uniform keys (full-head pass)"
    kidx = torch.as_tensor(_row_of_position(keys, S, N), device=DEV)
    dk_s = dk[b, h, kidx].double().cpu().numpy()
    dv_s = dv[b, h, kidx].double().cpu().numpy()
    args = [x[n][b, h].double().numpy() for n in ("q", "k", "v", "do")]
    t_keys = time.perf_counter()
    dk_ref, dv_ref = oracle.bwd_keys(*args, scale, keys)
    t_keys = time.perf_counter() - t_keys
    ek, ev = float(np.abs(dk_s - dk_ref).max()), float(np.abs(dv_s - dv_ref).max())
    early = keys < S // 8  # keys whose tiles see (almost) every query tile
    ek0 = float(np.abs(dk_s[early] - dk_ref[early]).max()) if early.any() else 0.0
    ev0 = float(np.abs(dv_s[early] - dv_ref[early]).max()) if early.any() else 0.0
    print(name, what, "max errors dk dv", ek, ev, "(first eighth:", ek0, ev0, ")",
          f"max |dk| {np.abs(dk_ref).max():.3f} |dv| {np.abs(dv_ref).max():.3f}",
          f"(oracle: {t_keys:.1f} s on {oracle.default_threads()} threads)")
    assert ek <= 2e-2 and ev <= 2e-2

    # invariants on every head and column (fp64 sums of the GPU tensors)
    pos = torch.as_tensor(oracle.layout_positions(S, N, sp.STRIPED), device=DEV)
    inv = grad_sum_errors(dv, dk, x["do"].to(DEV), x["q"].to(DEV), pos)
    print(name, "gradient invariants (max error, smallest bound, max error/bound):", inv)
    assert inv["dv"][2] <= 1.0 and inv["dk"][2] <= 1.0, inv


def test_mid_contiguous_and_per_round_sampled():
    """Mid workload (B=1, H=24, S=65536, N=8) in the contiguous placement
    (batched forward + backward) and through the per-round path (8 x 8
    ring_round_fwd calls merged in ring order), on 2048 sampled rows."""
    B, H, S, D, N = WORKLOADS["mid"]
    scale = 1.0 / D ** 0.5
    x = attention_inputs(B, H, S, D, torch.bfloat16, seed=1)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))  # contiguous = position order
    stats = sp.new_tile_stats(N, DEV)
    o, lse = sp.striped_attn_fwd(q, k, v, N, sp.CONTIGUOUS, tile_stats=stats)
    dq, dk, dv = sp.striped_attn_bwd(q, k, v, o, lse, do, N, sp.CONTIGUOUS)
    # per-round path on the striped layout
    qs, ks, vs = (sp.striped_permute(t, N) for t in (q, k, v))
    o_acc = torch.empty(B, H, S, D, dtype=torch.float32, device=DEV)
    lse_acc = torch.empty(B, H, S, dtype=torch.float32, device=DEV)
    rstats = sp.new_tile_stats(N, DEV)
    for d in range(N):
        for r in range(N):
            sp.ring_round_fwd(qs, ks, vs, o_acc, lse_acc, d, (d - r) % N, N, sp.STRIPED,
                              first_round=(r == 0), tile_stats=rstats)
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    full, part = oracle.tile_counts_closed(S, N, 128, sp.CONTIGUOUS)
    st = stats.cpu().numpy()
    assert np.array_equal(st[0], B * H * full) and np.array_equal(st[1], B * H * part)
    fs, ps = oracle.tile_counts_closed(S, N, 128, sp.STRIPED)
    rs = rstats.cpu().numpy()
    assert np.array_equal(rs[0], B * H * fs) and np.array_equal(rs[1], B * H * ps)

    rows = sample_rows(2048, B, H, S, seed=1).numpy()
    bidx, hidx = torch.as_tensor(rows[:, 0], device=DEV), torch.as_tensor(rows[:, 1], device=DEV)
    pidx = torch.as_tensor(rows[:, 2], device=DEV)
    sidx = torch.as_tensor(_row_of_position(rows[:, 2], S, N), device=DEV)
    got = {"o": o[bidx, hidx, pidx].double().cpu().numpy(), "lse": lse[bidx, hidx, pidx].double().cpu().numpy(),
           "dq": dq[bidx, hidx, pidx].double().cpu().numpy(),
           "o_round": o_acc[bidx, hidx, sidx].double().cpu().numpy(),
           "lse_round": lse_acc[bidx, hidx, sidx].double().cpu().numpy()}
    worst = dict.fromkeys(got, 0.0)
    for (b, h) in sorted({(int(r[0]), int(r[1])) for r in rows}):
        sel = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
        pos = rows[sel, 2]
        args = [x[n][b, h].double().numpy() for n in ("q", "k", "v", "do")]
        o_ref, lse_ref = oracle.attn_fwd(args[0], args[1], args[2], scale, rows=pos)
        _, _, dq_ref = oracle.bwd_rows(*args, scale, rows=pos)
        for key, ref in (("o", o_ref), ("lse", lse_ref), ("dq", dq_ref), ("o_round", o_ref),
                         ("lse_round", lse_ref)):
            worst[key] = max(worst[key], float(np.abs(got[key][sel] - ref).max()))
    print("mid contiguous / per-round max errors", worst)
    assert worst["o"] <= 2e-2 and worst["dq"] <= 2e-2 and worst["o_round"] <= 2e-2
    assert worst["lse"] <= 1e-3 and worst["lse_round"] <= 1e-3
    # gradient invariants of the contiguous backward on every head
    inv = grad_sum_errors(dv, dk, do, q, torch.arange(S, device=DEV))
    print("mid contiguous gradient invariants", inv)
    assert inv["dv"][2] <= 1.0 and inv["dk"][2] <= 1.0, inv


def test_mid_zigzag_sampled():
    """Mid workload (B=1, H=24, S=65536, N=8) in the zig-zag placement
    (permuted on the GPU): batched forward and backward on 2048 sampled
    query rows, per-round counters against the oracle's closed form, and
    the gradient invariants on every head."""
    B, H, S, D, N = WORKLOADS["mid"]
    scale = 1.0 / D ** 0.5
    x = attention_inputs(B, H, S, D, torch.bfloat16, seed=2)
    q, k, v, do = (sp.layout_permute(x[n].to(DEV), N, sp.ZIGZAG) for n in ("q", "k", "v", "do"))
    stats = sp.new_tile_stats(N, DEV)
    o, lse = sp.striped_attn_fwd(q, k, v, N, sp.ZIGZAG, tile_stats=stats)
    dq, dk, dv = sp.striped_attn_bwd(q, k, v, o, lse, do, N, sp.ZIGZAG)
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    full, part = oracle.tile_counts_closed(S, N, 128, oracle.ZIGZAG)
    st = stats.cpu().numpy()
    assert np.array_equal(st[0], B * H * full) and np.array_equal(st[1], B * H * part)
    rows = sample_rows(2048, B, H, S, seed=2).numpy()
    inv = np.empty(S, dtype=np.int64)
    inv[oracle.zigzag_positions(S, N)] = np.arange(S)  # position -> zig-zag row
    bidx, hidx = torch.as_tensor(rows[:, 0], device=DEV), torch.as_tensor(rows[:, 1], device=DEV)
    zidx = torch.as_tensor(inv[rows[:, 2]], device=DEV)
    got = {"o": o[bidx, hidx, zidx].double().cpu().numpy(), "lse": lse[bidx, hidx, zidx].double().cpu().numpy(),
           "dq": dq[bidx, hidx, zidx].double().cpu().numpy()}
    worst = dict.fromkeys(got, 0.0)
    for (b, h) in sorted({(int(r[0]), int(r[1])) for r in rows}):
        sel = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
        pos = rows[sel, 2]
        args = [x[n][b, h].double().numpy() for n in ("q", "k", "v", "do")]
        o_ref, lse_ref = oracle.attn_fwd(args[0], args[1], args[2], scale, rows=pos)
        _, _, dq_ref = oracle.bwd_rows(*args, scale, rows=pos)
        for key, ref in (("o", o_ref), ("lse", lse_ref), ("dq", dq_ref)):
            worst[key] = max(worst[key], float(np.abs(got[key][sel] - ref).max()))
    print("mid zig-zag max errors", worst)
    assert worst["o"] <= 2e-2 and worst["dq"] <= 2e-2 and worst["lse"] <= 1e-3
    inv = grad_sum_errors(dv, dk, x["do"].to(DEV), x["q"].to(DEV),
                          torch.as_tensor(oracle.zigzag_positions(S, N), device=DEV))
    print("mid zig-zag gradient invariants", inv)
    assert inv["dv"][2] <= 1.0 and inv["dk"][2] <= 1.0, inv
