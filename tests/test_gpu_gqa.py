"""Grouped-query attention on the GPU (H query heads sharing Hkv key/value
heads; query head h reads key/value head h // (H/Hkv)) against the fp64
oracle's per-head composition: O, LSE, dQ, and dK/dV summed over each
group, all three placements, with the per-round tile counters (counted per
query head) against the oracle's brute force.

Tolerance: O, LSE and dQ are per query head and keep the multi-head bounds.
dK and dV of a shared head are sums of G = H/Hkv per-head gradients, each
with the multi-head error (bf16 rounding of P and dS as tensor-core
operands); independent errors of G terms add up to about sqrt(G) times one
term's, so their bound is the multi-head one times sqrt(G)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs, sample_rows, sample_tail_keys
from tests._util import TOL, grad_sum_errors, maxerr, to_layout, to_positions

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _gqa_inputs(B, H, Hkv, S, D, dtype, seed):
    """Seeded inputs: q, dO with H heads; k, v with Hkv heads (the first Hkv
    heads of a second H-head draw)."""
    x = attention_inputs(B, H, S, D, dtype, seed=seed)
    y = attention_inputs(B, H, S, D, dtype, seed=seed + 100, with_do=False)
    return {"q": x["q"], "do": x["do"], "k": y["k"][:, :Hkv].contiguous(), "v": y["v"][:, :Hkv].contiguous()}


CASES = [
    # dtype, B, H, Hkv, S, D, N, layouts
    (torch.float32, 1, 4, 2, 256, 64, 4, (sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG)),
    (torch.float32, 2, 4, 1, 128, 32, 4, (sp.STRIPED, sp.ZIGZAG)),
    (torch.bfloat16, 1, 4, 2, 1024, 128, 4, (sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG)),
    (torch.bfloat16, 1, 8, 2, 2048, 128, 8, (sp.STRIPED, sp.ZIGZAG)),
    (torch.bfloat16, 2, 6, 3, 1200, 128, 4, (sp.STRIPED, sp.CONTIGUOUS)),  # ragged stripe tail
    (torch.bfloat16, 1, 4, 1, 8192, 128, 8, (sp.STRIPED,)),
    (torch.bfloat16, 1, 4, 2, 2048, 64, 4, (sp.STRIPED, sp.ZIGZAG)),  # head dimension 64
]


@pytest.mark.parametrize("dtype,B,H,Hkv,S,D,N,layouts", CASES)
def test_gqa_fwd_bwd_match_oracle(dtype, B, H, Hkv, S, D, N, layouts):
    x = _gqa_inputs(B, H, Hkv, S, D, dtype, seed=21)
    scale = 1.0 / D ** 0.5
    ref = {}
    for b in range(B):
        args = [x[n][b].double().numpy() for n in ("q", "k", "v", "do")]
        ref[b] = (oracle.attn_fwd_gqa(args[0], args[1], args[2], scale), oracle.attn_bwd_gqa(*args, scale))
    tol = TOL[dtype]
    T = sp.kernel_tile(dtype, D)
    for layout in layouts:
        q, k, v, do = (to_layout(x[n], N, layout, DEV) for n in ("q", "k", "v", "do"))
        fst, bst = sp.new_tile_stats(N, DEV), sp.new_tile_stats(N, DEV)
        o, lse = sp.striped_attn_fwd_gqa(q, k, v, N, layout, tile_stats=fst)
        dq, dk, dv = sp.striped_attn_bwd_gqa(q, k, v, o, lse, do, N, layout, tile_stats=bst)
        assert dk.shape == k.shape and dv.shape == v.shape
        torch.cuda.synchronize()
        assert sp.check_error() == 0
        got = {n: to_positions(t, N, layout) for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
        lse_pos = to_positions(lse[..., None], N, layout)[..., 0]
        for b in range(B):
            (o_r, l_r), (dq_r, dk_r, dv_r) = ref[b]
            assert maxerr(got["o"][b], o_r) <= tol["o"], layout
            assert maxerr(lse_pos[b], l_r) <= tol["lse"], layout
            kv_tol = tol["grad"] * np.sqrt(H // Hkv)
            for n, r, t in (("dq", dq_r, tol["grad"]), ("dk", dk_r, kv_tol), ("dv", dv_r, kv_tol)):
                assert maxerr(got[n][b], r) <= t, (layout, n, maxerr(got[n][b], r))
        full, part = oracle.tile_counts_bruteforce(S, N, T, T, layout)
        for st in (fst, bst):
            c = st.cpu().numpy()
            assert np.array_equal(c[0], B * H * full) and np.array_equal(c[1], B * H * part)


def test_gqa_group_of_one_equals_mha():
    """Hkv = H through the grouped entry points is bit-identical to the
    plain ones (same kernels, G = 1)."""
    B, H, S, D, N = 1, 2, 1024, 128, 4
    x = attention_inputs(B, H, S, D, torch.bfloat16, seed=23)
    q, k, v, do = (to_layout(x[n], N, sp.STRIPED, DEV) for n in ("q", "k", "v", "do"))
    o1, l1 = sp.striped_attn_fwd(q, k, v, N)
    o2, l2 = sp.striped_attn_fwd_gqa(q, k, v, N)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = sp.striped_attn_bwd(q, k, v, o1, l1, do, N)
    g2 = sp.striped_attn_bwd_gqa(q, k, v, o1, l1, do, N)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert maxerr(g1[0].float().cpu(), g2[0].float().cpu()) <= 1e-2  # dQ: fp32 atomics, order varies


@pytest.mark.slow
def test_gqa_mid_size_sampled():
    """Mid workload shape with grouped K/V (B=1, H=24, Hkv=8, S=65536,
    D=128, N=8, striped): 2048 sampled query rows for O, LSE, dQ; dK and dV
    of 128 key positions from the tail of one key/value head, each the sum
    over its 3 query heads; the dV invariant sum_t dV_t = sum over the group
    of sum_p dO_p on every key/value head."""
    B, H, Hkv, S, D, N = 1, 24, 8, 65536, 128, 8
    G = H // Hkv
    scale = 1.0 / D ** 0.5
    x = _gqa_inputs(B, H, Hkv, S, D, torch.bfloat16, seed=24)
    q, k, v, do = (sp.striped_permute(x[n].to(DEV), N) for n in ("q", "k", "v", "do"))
    o, lse = sp.striped_attn_fwd_gqa(q, k, v, N)
    dq, dk, dv = sp.striped_attn_bwd_gqa(q, k, v, o, lse, do, N)
    torch.cuda.synchronize()
    assert sp.check_error() == 0
    L = S // N
    srow = lambda p: (p % N) * L + p // N  # noqa: E731  (striped row of position p)
    rows = sample_rows(2048, B, H, S, seed=24).numpy()
    idx = torch.as_tensor(srow(rows[:, 2]), device=DEV)
    hidx = torch.as_tensor(rows[:, 1], device=DEV)
    got = {"o": o[0, hidx, idx].double().cpu().numpy(), "lse": lse[0, hidx, idx].double().cpu().numpy(),
           "dq": dq[0, hidx, idx].double().cpu().numpy()}
    worst = dict.fromkeys(got, 0.0)
    for h in sorted({int(r[1]) for r in rows}):
        sel = np.nonzero(rows[:, 1] == h)[0]
        pos = rows[sel, 2]
        args = [x["q"][0, h], x["k"][0, h // G], x["v"][0, h // G], x["do"][0, h]]
        args = [t.double().numpy() for t in args]
        o_r, l_r = oracle.attn_fwd(args[0], args[1], args[2], scale, rows=pos)
        _, _, dq_r = oracle.bwd_rows(*args, scale, rows=pos)
        for n, r in (("o", o_r), ("lse", l_r), ("dq", dq_r)):
            worst[n] = max(worst[n], float(np.abs(got[n][sel] - r).max()))
    print("gqa mid sampled max errors", worst)
    assert worst["o"] <= 2e-2 and worst["dq"] <= 2e-2 and worst["lse"] <= 1e-3
    kvh = 5
    keys = sample_tail_keys(128, S, 1024, seed=24).numpy()
    dk_r = np.zeros((len(keys), D))
    dv_r = np.zeros((len(keys), D))
    for h in range(kvh * G, (kvh + 1) * G):
        args = [x["q"][0, h], x["k"][0, kvh], x["v"][0, kvh], x["do"][0, h]]
        gk, gv = oracle.bwd_keys(*[t.double().numpy() for t in args], scale, keys)
        dk_r += gk
        dv_r += gv
    kidx = torch.as_tensor(srow(keys), device=DEV)
    ek = float(np.abs(dk[0, kvh, kidx].double().cpu().numpy() - dk_r).max())
    ev = float(np.abs(dv[0, kvh, kidx].double().cpu().numpy() - dv_r).max())
    print("gqa mid tail-key max errors dk dv", ek, ev)
    assert ek <= 2e-2 * np.sqrt(G) and ev <= 2e-2 * np.sqrt(G)
    pos = torch.as_tensor(oracle.layout_positions(S, N, sp.STRIPED), device=DEV)
    inv = grad_sum_errors(dv, dk, x["do"].to(DEV), x["q"].to(DEV), pos, G=G)
    print("gqa mid gradient invariants", inv)
    assert inv["dv"][2] <= 1.0 and inv["dk"][2] <= 1.0, inv
