"""Packed variable-length batches on the GPU: the packed permutation
bit-exact against the oracle's per-sequence placement, and the forward and
backward (with and without grouped K/V heads) against the oracle's
per-sequence attention, all three placements, fp32 and bf16, with the tile
counters equal to the sum of the sequences' own tables.  bf16 dK and dV are
compared after allowing each element the rounding of its own stored bf16
value (half an ulp at that element), so the 2e-2 bound applies to the
arithmetic before storage (dK/dV of a packed D = 64 head reach |dV| ~ 4.8,
where stored bf16 values lie 2^-5 apart)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs
from tests._util import TOL, bf16_storage_excess, maxerr

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N,cu", [(4, [0, 8, 40, 48, 128]), (8, [0, 64, 80, 1024]), (1, [0, 2, 3, 10])])
def test_varlen_permute_bit_exact(N, cu, dtype, layout):
    if layout == sp.ZIGZAG and any((b - a) % (2 * N) for a, b in zip(cu, cu[1:])):
        pytest.skip("zig-zag needs every length a multiple of 2N")
    H, D = 3, 64
    S = cu[-1]
    x = torch.randn(H, S, D, generator=torch.Generator().manual_seed(7)).to(dtype)
    pos = torch.as_tensor(oracle.varlen_positions(cu, N, layout))
    y = sp.striped_varlen_permute(x.to(DEV), cu, N, layout)
    assert torch.equal(y.cpu(), x[:, pos])
    assert torch.equal(sp.striped_varlen_unpermute(y, cu, N, layout).cpu(), x)


def _inputs(H, Hkv, S, D, dtype, seed):
    x = attention_inputs(1, H, S, D, dtype, seed=seed)
    y = attention_inputs(1, H, S, D, dtype, seed=seed + 50, with_do=False)
    return {"q": x["q"][0], "do": x["do"][0], "k": y["k"][0, :Hkv].contiguous(), "v": y["v"][0, :Hkv].contiguous()}


CASES = [
    # dtype, H, Hkv, D, N, cu_seqlens, layouts
    (torch.float32, 2, 2, 64, 4, [0, 64, 192, 256, 448], (sp.STRIPED, sp.CONTIGUOUS)),
    (torch.float32, 4, 2, 32, 4, [0, 128, 384, 512], (sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG)),
    (torch.bfloat16, 2, 2, 128, 4, [0, 512, 2048, 2560, 4096], (sp.STRIPED, sp.CONTIGUOUS)),
    (torch.bfloat16, 4, 2, 128, 4, [0, 1024, 3072, 4096], (sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG)),
    (torch.bfloat16, 2, 1, 128, 8, [0, 2048, 3072, 8192], (sp.STRIPED, sp.CONTIGUOUS)),
    (torch.bfloat16, 2, 1, 128, 8, [0, 2048, 6144, 8192], (sp.ZIGZAG,)),  # zig-zag: multiples of 2N*T
    (torch.bfloat16, 2, 2, 64, 4, [0, 1024, 3072, 4096], (sp.STRIPED, sp.ZIGZAG)),  # head dimension 64
]


@pytest.mark.parametrize("dtype,H,Hkv,D,N,cu,layouts", CASES)
def test_varlen_fwd_bwd_match_oracle(dtype, H, Hkv, D, N, cu, layouts):
    S = cu[-1]
    G = H // Hkv
    x = _inputs(H, Hkv, S, D, dtype, seed=31)
    scale = 1.0 / D ** 0.5
    ref_o, ref_l, ref_dq = [], [], []
    ref_dk = np.zeros((Hkv, S, D))
    ref_dv = np.zeros((Hkv, S, D))
    for h in range(H):
        q, k, v, do = (t.double().numpy() for t in (x["q"][h], x["k"][h // G], x["v"][h // G], x["do"][h]))
        o, l = oracle.attn_fwd_varlen(q, k, v, cu, scale)
        gq, gk, gv = oracle.attn_bwd_varlen(q, k, v, do, cu, scale)
        ref_o.append(o)
        ref_l.append(l)
        ref_dq.append(gq)
        ref_dk[h // G] += gk
        ref_dv[h // G] += gv
    tol = TOL[dtype]
    T = sp.kernel_tile(dtype, D)
    for layout in layouts:
        pos = oracle.varlen_positions(cu, N, layout)
        q, k, v, do = (sp.striped_varlen_permute(x[n].to(DEV), cu, N, layout) for n in ("q", "k", "v", "do"))
        fst, bst = sp.new_tile_stats(N, DEV), sp.new_tile_stats(N, DEV)
        o, lse = sp.striped_attn_fwd_varlen(q, k, v, cu, N, layout, tile_stats=fst)
        dq, dk, dv = sp.striped_attn_bwd_varlen(q, k, v, o, lse, do, cu, N, layout, tile_stats=bst)
        torch.cuda.synchronize()
        assert sp.check_error() == 0

        def back(t):  # layout rows -> positions, float64 numpy
            a = t.double().cpu().numpy()
            out = np.empty_like(a)
            out[:, pos] = a
            return out

        o_p, l_p, dq_p, dk_p, dv_p = back(o), back(lse), back(dq), back(dk), back(dv)
        kv_tol = tol["grad"] * np.sqrt(G)
        bf = dtype == torch.bfloat16
        for h in range(H):
            assert maxerr(o_p[h], ref_o[h]) <= tol["o"], (layout, h)
            assert maxerr(l_p[h], ref_l[h]) <= tol["lse"], (layout, h)
            assert maxerr(dq_p[h], ref_dq[h]) <= tol["grad"], (layout, h)
        err = bf16_storage_excess if bf else maxerr
        assert err(dk_p, ref_dk) <= kv_tol, (layout, err(dk_p, ref_dk), maxerr(dk_p, ref_dk))
        assert err(dv_p, ref_dv) <= kv_tol, (layout, err(dv_p, ref_dv), maxerr(dv_p, ref_dv))
        full = sum(oracle.tile_counts_bruteforce(b - a, N, T, T, layout)[0] for a, b in zip(cu, cu[1:]))
        part = sum(oracle.tile_counts_bruteforce(b - a, N, T, T, layout)[1] for a, b in zip(cu, cu[1:]))
        for st in (fst, bst):
            c = st.cpu().numpy()
            assert np.array_equal(c[0], H * full) and np.array_equal(c[1], H * part), layout


def test_varlen_single_sequence_equals_dense():
    """One packed sequence is the dense call: identical O, LSE, dK, dV."""
    H, S, D, N = 2, 2048, 128, 8
    x = attention_inputs(1, H, S, D, torch.bfloat16, seed=33)
    q, k, v, do = (sp.striped_permute(x[n].to(DEV), N) for n in ("q", "k", "v", "do"))
    o1, l1 = sp.striped_attn_fwd(q, k, v, N)
    o2, l2 = sp.striped_attn_fwd_varlen(q[0], k[0], v[0], [0, S], N)
    assert torch.equal(o1[0], o2) and torch.equal(l1[0], l2)
    g1 = sp.striped_attn_bwd(q, k, v, o1, l1, do, N)
    g2 = sp.striped_attn_bwd_varlen(q[0], k[0], v[0], o2, l2, do[0], [0, S], N)
    assert torch.equal(g1[1][0], g2[1]) and torch.equal(g1[2][0], g2[2])
    assert maxerr(g1[0][0].float().cpu(), g2[0].float().cpu()) <= 1e-2
