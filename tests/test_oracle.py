"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: a library
routine (torch's fp64 causal scaled-dot-product attention and its autograd,
scipy's logsumexp), closed forms and special cases of the definition,
central finite differences, invariants, and brute force on tiny inputs.
A plausible slip in the oracle (dropped term, wrong sign, off-by-one in the
causal bound, transposed operand, wrong stripe index) fails at least one.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from oracle import CONTIGUOUS, STRIPED, ZIGZAG


def _rand(S, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((S, D)) * scale


def _sdpa(q, k, v):
    """torch's fp64 causal attention on the CPU (a library routine)."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=True)[0, 0].numpy()


# ---------------------------------------------------------------- placement
@pytest.mark.parametrize("S,N", [(8, 1), (8, 2), (12, 4), (256, 4), (64, 8), (48, 16)])
def test_stripe_positions_every_nth_token(oracle_lib, S, N):
    """Stripe d holds exactly the positions p with p mod N == d, ascending
    ("every N-th token"), and the map is a permutation."""
    L = S // N
    pos = oracle.stripe_positions(S, N)
    assert sorted(pos.tolist()) == list(range(S))
    for d in range(N):
        stripe = pos[d * L:(d + 1) * L]
        assert all(p % N == d for p in stripe)
        assert np.all(np.diff(stripe) == N)
    for row in range(S):
        assert oracle.position_of_row(row, S, N, STRIPED) == pos[row]
        assert oracle.position_of_row(row, S, N, CONTIGUOUS) == row


def test_stripe_positions_n1_is_identity(oracle_lib):
    assert np.array_equal(oracle.stripe_positions(40, 1), np.arange(40))


@pytest.mark.parametrize("S,N", [(8, 1), (8, 2), (16, 4), (256, 4), (64, 8), (96, 16)])
def test_zigzag_positions_one_chunk_from_each_end(oracle_lib, S, N):
    """Device d holds chunk d, then chunk 2N-1-d, each ascending and whole
    (chunks of S/(2N)); the map is a permutation and position_of_row agrees
    with the enumeration."""
    L, C = S // N, S // (2 * N)
    pos = oracle.zigzag_positions(S, N)
    assert sorted(pos.tolist()) == list(range(S))
    for d in range(N):
        dev = pos[d * L:(d + 1) * L]
        assert dev[:C].tolist() == list(range(d * C, (d + 1) * C))
        assert dev[C:].tolist() == list(range((2 * N - 1 - d) * C, (2 * N - d) * C))
    for row in range(S):
        assert oracle.position_of_row(row, S, N, ZIGZAG) == pos[row]
    assert np.array_equal(oracle.layout_positions(S, N, ZIGZAG), pos)


def test_zigzag_n1_is_identity(oracle_lib):
    assert np.array_equal(oracle.zigzag_positions(40, 1), np.arange(40))


# ---------------------------------------------------------------- forward
@pytest.mark.parametrize("S,D", [(1, 4), (7, 3), (33, 16), (64, 64)])
def test_fwd_matches_torch_sdpa(oracle_lib, S, D):
    q, k, v = _rand(S, D, 1), _rand(S, D, 2), _rand(S, D, 3)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attn_fwd(q, k, v, scale)
    assert np.allclose(o, _sdpa(q, k, v), atol=1e-12, rtol=1e-12)
    # LSE against scipy's logsumexp of each causal score row
    s = scale * q @ k.T
    ref = np.array([logsumexp(s[p, :p + 1]) for p in range(S)])
    assert np.allclose(lse, ref, atol=1e-12, rtol=1e-12)


def test_fwd_naive_triple_loop(oracle_lib):
    """Direct loops, no max subtraction, on a tiny input."""
    S, D = 9, 5
    q, k, v = _rand(S, D, 4, 0.5), _rand(S, D, 5, 0.5), _rand(S, D, 6)
    scale = 0.7
    o, lse = oracle.attn_fwd(q, k, v, scale)
    for p in range(S):
        w = [math.exp(scale * sum(q[p, c] * k[t, c] for c in range(D))) for t in range(p + 1)]
        z = sum(w)
        assert abs(lse[p] - math.log(z)) < 1e-12
        for c in range(D):
            assert abs(o[p, c] - sum(w[t] * v[t, c] for t in range(p + 1)) / z) < 1e-12


def test_first_position_attends_only_itself(oracle_lib):
    S, D = 50, 16
    q, k, v = _rand(S, D, 7), _rand(S, D, 8), _rand(S, D, 9)
    scale = 0.25
    o, lse = oracle.attn_fwd(q, k, v, scale)
    assert np.allclose(o[0], v[0], atol=1e-14)
    assert abs(lse[0] - scale * q[0] @ k[0]) < 1e-13


def test_constant_keys_give_prefix_mean(oracle_lib):
    """All keys equal -> uniform weights over t <= p: O_p is the prefix mean
    of v and LSE_p = s<q_p, k> + log(p + 1)."""
    S, D = 40, 8
    q, v = _rand(S, D, 10), _rand(S, D, 11)
    k = np.tile(_rand(1, D, 12), (S, 1))
    scale = 0.3
    o, lse = oracle.attn_fwd(q, k, v, scale)
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    assert np.allclose(o, prefix_mean, atol=1e-12)
    assert np.allclose(lse, scale * q @ k[0] + np.log(np.arange(1, S + 1)), atol=1e-12)


def test_rows_of_p_sum_to_one(oracle_lib):
    """V = 1 everywhere -> every output entry is sum_t P_pt = 1."""
    S, D = 30, 6
    q, k = _rand(S, D, 13, 2.0), _rand(S, D, 14, 2.0)
    o, _ = oracle.attn_fwd(q, k, np.ones((S, D)), 0.5)
    assert np.allclose(o, 1.0, atol=1e-13)


def test_key_shift_invariance(oracle_lib):
    """k_t -> k_t + c shifts score row p by s<q_p, c>: O unchanged, LSE
    shifted by exactly that amount."""
    S, D = 45, 12
    q, k, v = _rand(S, D, 15), _rand(S, D, 16), _rand(S, D, 17)
    c = _rand(1, D, 18)[0]
    scale = 0.4
    o1, l1 = oracle.attn_fwd(q, k, v, scale)
    o2, l2 = oracle.attn_fwd(q, k + c, v, scale)
    assert np.allclose(o1, o2, atol=1e-12)
    assert np.allclose(l2 - l1, scale * q @ c, atol=1e-12)


def test_selected_rows_match_all_rows(oracle_lib):
    S, D = 70, 8
    q, k, v = _rand(S, D, 19), _rand(S, D, 20), _rand(S, D, 21)
    o, lse = oracle.attn_fwd(q, k, v, 0.3)
    rows = np.array([69, 0, 13, 13, 42])
    o2, lse2 = oracle.attn_fwd(q, k, v, 0.3, rows=rows)
    assert np.array_equal(o2, o[rows]) and np.array_equal(lse2, lse[rows])


@pytest.mark.parametrize("layout", [STRIPED, CONTIGUOUS, ZIGZAG])
def test_round_partials_merge_to_full(oracle_lib, layout):
    """Per-round partial results over each device's key set, merged with the
    log-sum-exp rule in ring order, reproduce full causal attention."""
    S, D, N = 48, 8, 4
    L = S // N
    q, k, v = _rand(S, D, 22), _rand(S, D, 23), _rand(S, D, 24)
    scale = 0.35
    o_full, lse_full = oracle.attn_fwd(q, k, v, scale)
    for d in range(N):
        rows = np.array([oracle.position_of_row(d * L + i, S, N, layout) for i in range(L)])
        acc_o = acc_l = None
        for r in range(N):
            e = (d - r) % N
            keyset = np.zeros(S, dtype=bool)
            for j in range(L):
                keyset[oracle.position_of_row(e * L + j, S, N, layout)] = True
            o_r, l_r = oracle.attn_fwd(q, k, v, scale, rows=rows, key_in_set=keyset)
            if acc_o is None:
                acc_o, acc_l = o_r, l_r
            else:
                acc_o, acc_l = oracle.merge_rounds(acc_o, acc_l, o_r, l_r)
        assert np.allclose(acc_o, o_full[rows], atol=1e-12)
        assert np.allclose(acc_l, lse_full[rows], atol=1e-12)


def test_empty_key_set(oracle_lib):
    S, D = 10, 4
    q, k, v = _rand(S, D, 25), _rand(S, D, 26), _rand(S, D, 27)
    keyset = np.zeros(S, dtype=bool)
    keyset[5:] = True  # rows 0..4 see no key
    o, lse = oracle.attn_fwd(q, k, v, 1.0, key_in_set=keyset)
    assert np.all(np.isneginf(lse[:5])) and np.all(o[:5] == 0)
    assert np.all(np.isfinite(lse[5:]))


# ---------------------------------------------------------------- backward
@pytest.mark.parametrize("S,D", [(1, 3), (6, 4), (37, 16), (64, 32)])
def test_bwd_matches_torch_autograd(oracle_lib, S, D):
    q, k, v, do = (_rand(S, D, 30 + i) for i in range(4))
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=True)[0, 0]
    out.backward(torch.tensor(do))
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_bwd_central_finite_differences(oracle_lib):
    """d/dx of L = sum <dO, O> by central differences of the oracle forward."""
    S, D = 7, 3
    q, k, v, do = (_rand(S, D, 40 + i) for i in range(4))
    scale = 0.6
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, scale, nthreads=1)
        return float(np.sum(o * do))

    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        for p in range(S):
            for c in range(D):
                args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                args[name][p, c] += h
                up = loss(args["q"], args["k"], args["v"])
                args[name][p, c] -= 2 * h
                dn = loss(args["q"], args["k"], args["v"])
                assert abs((up - dn) / (2 * h) - grad[p, c]) < 1e-7, (name, p, c)


def test_bwd_invariants(oracle_lib):
    """sum_t dV_t = sum_p dO_p (rows of P sum to 1) and sum_t dK_t = 0
    (each row of dS sums to 0); dQ_0 = 0 (dS_00 = 0: one kept key)."""
    S, D = 80, 16
    q, k, v, do = (_rand(S, D, 50 + i) for i in range(4))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.25)
    assert np.allclose(dv.sum(0), do.sum(0), atol=1e-11)
    assert np.allclose(dk.sum(0), 0.0, atol=1e-11)
    assert np.allclose(dq[0], 0.0, atol=1e-14)


def test_bwd_J_equals_dO_dot_O(oracle_lib):
    S, D = 50, 8
    q, k, v, do = (_rand(S, D, 60 + i) for i in range(4))
    lse, J, _ = oracle.bwd_rows(q, k, v, do, 0.3, want_dq=False)
    o, lse2 = oracle.attn_fwd(q, k, v, 0.3)
    assert np.allclose(J, np.sum(do * o, axis=1), atol=1e-12)
    assert np.allclose(lse, lse2, atol=1e-13)


def test_bwd_sampled_keys_match_full(oracle_lib):
    S, D = 90, 8
    q, k, v, do = (_rand(S, D, 70 + i) for i in range(4))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.3)
    keys = np.array([89, 60, 71, 75])
    dk2, dv2 = oracle.bwd_keys(q, k, v, do, 0.3, keys)
    assert np.allclose(dk2, dk[keys], atol=1e-13) and np.allclose(dv2, dv[keys], atol=1e-13)
    rows = np.array([3, 89, 45])
    _, _, dq2 = oracle.bwd_rows(q, k, v, do, 0.3, rows=rows)
    assert np.allclose(dq2, dq[rows], atol=1e-13)


# ---------------------------------------------------------------- tiles
@pytest.mark.parametrize("layout", [STRIPED, CONTIGUOUS])
@pytest.mark.parametrize("S,N,T", [(16, 1, 4), (64, 4, 4), (256, 4, 16), (256, 4, 64),
                                   (96, 8, 3), (128, 8, 1), (8192, 8, 128), (64, 2, 2)])
def test_tile_counts_bruteforce_equals_closed_form(oracle_lib, S, N, T, layout):
    bf = oracle.tile_counts_bruteforce(S, N, T, T, layout)
    cf = oracle.tile_counts_closed(S, N, T, layout)
    assert np.array_equal(bf[0], cf[0]) and np.array_equal(bf[1], cf[1])


@pytest.mark.parametrize("S,N,T", [(16, 1, 4), (64, 4, 4), (256, 4, 16), (256, 4, 32), (96, 8, 3),
                                   (128, 8, 1), (8192, 8, 128), (64, 2, 2), (1536, 12, 64)])
def test_zigzag_bruteforce_equals_closed_form(oracle_lib, S, N, T):
    bf = oracle.tile_counts_bruteforce(S, N, T, T, ZIGZAG)
    cf = oracle.tile_counts_closed(S, N, T, ZIGZAG)
    assert np.array_equal(bf[0], cf[0]) and np.array_equal(bf[1], cf[1])


def test_zigzag_rounds_balanced_without_diagonals(oracle_lib):
    """Zig-zag: after round 0 every device keeps exactly two whole chunk
    pairs (2c^2 full tiles, no partial tile); round 0 is two causal chunk
    triangles plus one whole chunk pair (2c^2 + c tiles, 2c of them
    partial).  Its total equals the contiguous placement's."""
    S, N, T = 8192, 8, 128
    c = S // (2 * N) // T
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, ZIGZAG)
    assert np.all(part[1:] == 0) and np.all(full[1:] == 2 * c * c)
    assert np.all(full[0] + part[0] == 2 * c * c + c) and np.all(part[0] == 2 * c)
    cf, cp = oracle.tile_counts_bruteforce(S, N, T, T, CONTIGUOUS)
    assert full.sum() + part.sum() == cf.sum() + cp.sum()


def test_striped_rounds_skip_about_half(oracle_lib):
    """Striped: every device does the same work in every round, about half
    of the n^2 tiles of the round (the balance claim)."""
    S, N, T = 8192, 8, 128
    n = S // N // T
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, STRIPED)
    work = full + part
    assert np.all(work == work[0, 0])
    assert work[0, 0] == n * (n + 1) // 2
    assert abs(work[0, 0] / n ** 2 - 0.5) <= 1.0 / n


def test_contiguous_rounds_all_or_nothing(oracle_lib):
    """Contiguous: after round 0 each device's round is fully kept or fully
    skipped (the imbalance claim); round 0 is the causal triangle."""
    S, N, T = 4096, 8, 64
    n = S // N // T
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, CONTIGUOUS)
    assert np.all(full[0] + part[0] == n * (n + 1) // 2)
    for r in range(1, N):
        for d in range(N):
            e = (d - r) % N
            assert part[r, d] == 0
            assert full[r, d] == (n * n if e < d else 0)


def test_ragged_tail_tiles(oracle_lib):
    """L = 2T + 1: the last striped diagonal tile is a single pair (i, i),
    kept iff e <= d; so it is full for e <= d and absent for e > d."""
    T, N = 4, 4
    L = 2 * T + 1
    S = N * L
    full, part = oracle.tile_counts_bruteforce(S, N, T, T, STRIPED)
    for r in range(N):
        for d in range(N):
            e = (d - r) % N
            # tiles: rows {0..3},{4..7},{8}; below diagonal 3 full; 2 partial diagonals
            assert part[r, d] == 2
            assert full[r, d] == 3 + (1 if e <= d else 0)


def test_critical_path_values(oracle_lib):
    """Critical path: striped N * n(n+1)/2; contiguous n(n+1)/2 + (N-1) n^2."""
    for S, N, T in [(256, 4, 16), (8192, 8, 128), (65536, 8, 128)]:
        n = S // N // T
        cp_s = oracle.critical_path(*oracle.tile_counts_closed(S, N, T, STRIPED))
        cp_c = oracle.critical_path(*oracle.tile_counts_closed(S, N, T, CONTIGUOUS))
        assert cp_s == N * n * (n + 1) // 2
        assert cp_c == n * (n + 1) // 2 + (N - 1) * n * n
    bf = oracle.tile_counts_bruteforce(256, 4, 16, 16, STRIPED)
    assert oracle.critical_path(*bf) == 40
    bf = oracle.tile_counts_bruteforce(256, 4, 16, 16, CONTIGUOUS)
    assert oracle.critical_path(*bf) == 58


def test_zigzag_critical_path(oracle_lib):
    """Zig-zag critical path 2N c^2 + c (c = S/(2N)/T): below the striped
    N n(n+1)/2 = 2N c^2 + N c by the (N-1) c diagonal tiles striped adds."""
    for S, N, T in [(256, 4, 16), (8192, 8, 128), (262144, 8, 128), (786432, 16, 128)]:
        c = S // (2 * N) // T
        cp_z = oracle.critical_path(*oracle.tile_counts_closed(S, N, T, ZIGZAG))
        cp_s = oracle.critical_path(*oracle.tile_counts_closed(S, N, T, STRIPED))
        assert cp_z == 2 * N * c * c + c
        assert cp_s - cp_z == (N - 1) * c
    assert oracle.critical_path(*oracle.tile_counts_bruteforce(256, 4, 16, 16, ZIGZAG)) == 2 * 4 * 4 + 2


def test_kept_pairs_equal_causal_total(oracle_lib):
    """With T = 1 every kept pair is one full tile: the total over rounds and
    devices is S(S+1)/2 for both placements."""
    S, N = 96, 8
    for layout in (STRIPED, CONTIGUOUS, ZIGZAG):
        full, part = oracle.tile_counts_bruteforce(S, N, 1, 1, layout)
        assert part.sum() == 0 and full.sum() == S * (S + 1) // 2


# ---------------------------------------------------------------- grouped-query attention
@pytest.mark.parametrize("H,Hkv", [(2, 2), (4, 2), (4, 1), (6, 2)])
def test_gqa_matches_torch_autograd_with_repeated_kv(oracle_lib, H, Hkv):
    """torch's fp64 causal SDPA on K/V repeated to every query head of its
    group (repeat_interleave), differentiated by autograd: the gradient of a
    shared head is what autograd accumulates through the repeat."""
    S, D = 24, 8
    rng = np.random.default_rng(40 + H + Hkv)
    q = rng.standard_normal((H, S, D))
    k = rng.standard_normal((Hkv, S, D))
    v = rng.standard_normal((Hkv, S, D))
    do = rng.standard_normal((H, S, D))
    scale = 0.4
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    G = H // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk.repeat_interleave(G, dim=0)[None], tv.repeat_interleave(G, dim=0)[None],
        is_causal=True, scale=scale)[0]
    o.backward(torch.tensor(do))
    o_ref, _ = oracle.attn_fwd_gqa(q, k, v, scale)
    assert np.allclose(o_ref, o.detach().numpy(), atol=1e-12)
    dq, dk, dv = oracle.attn_bwd_gqa(q, k, v, do, scale)
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)


# ---------------------------------------------------------------- packed variable-length batches
def test_varlen_matches_torch_block_diagonal_mask(oracle_lib):
    """Packed sequences: torch's fp64 SDPA with an explicit block-diagonal
    causal mask (keep t <= p inside one sequence), and its autograd."""
    cu = [0, 8, 24, 28, 48]
    S, D = cu[-1], 6
    rng = np.random.default_rng(51)
    q, k, v, do = (rng.standard_normal((S, D)) for _ in range(4))
    seq = np.repeat(np.arange(len(cu) - 1), np.diff(cu))
    keep = (seq[:, None] == seq[None, :]) & (np.arange(S)[None, :] <= np.arange(S)[:, None])
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                         attn_mask=torch.tensor(keep), scale=0.3)[0, 0]
    o.backward(torch.tensor(do))
    o_ref, _ = oracle.attn_fwd_varlen(q, k, v, cu, 0.3)
    assert np.allclose(o_ref, o.detach().numpy(), atol=1e-12)
    g = oracle.attn_bwd_varlen(q, k, v, do, cu, 0.3)
    for got, t in zip(g, (tq, tk, tv)):
        assert np.allclose(got, t.grad.numpy(), atol=1e-11)


@pytest.mark.parametrize("layout", [STRIPED, CONTIGUOUS, ZIGZAG])
def test_varlen_positions_place_each_sequence_on_its_own(oracle_lib, layout):
    """Every device's rows hold, sequence after sequence, that sequence's own
    placement; the map is a permutation; one sequence reduces to the plain
    placement."""
    N = 4
    cu = [0, 16, 24, 56, 64]
    pos = oracle.varlen_positions(cu, N, layout)
    S = cu[-1]
    assert sorted(pos.tolist()) == list(range(S))
    L = S // N
    for d in range(N):
        rows = pos[d * L:(d + 1) * L]
        off = 0
        for i in range(len(cu) - 1):
            Li = (cu[i + 1] - cu[i]) // N
            own = oracle.layout_positions(cu[i + 1] - cu[i], N, layout)[d * Li:(d + 1) * Li]
            assert np.array_equal(rows[off:off + Li], cu[i] + own)
            off += Li
    assert np.array_equal(oracle.varlen_positions([0, 64], N, layout), oracle.layout_positions(64, N, layout))


@pytest.mark.parametrize("layout", [STRIPED, CONTIGUOUS, ZIGZAG])
@pytest.mark.parametrize("N,cu", [(4, [0, 16, 24, 56, 64]), (2, [0, 4, 12, 20]), (8, [0, 16, 48, 64]),
                                  (1, [0, 3, 10])])
def test_varlen_positions_independent_enumeration(oracle_lib, N, cu, layout):
    """An enumeration written from the placement rules alone, position by
    position (no call into the oracle's placements): position p of sequence
    i (offset t = p - cu[i], length S_i, L_i = S_i / N rows per device) sits
    on device d at local row j of that sequence's block, which starts at row
    d*L + cu[i]/N of the packed head --
      striped:    every N-th token, d = t mod N, j = t div N
      contiguous: d = t div L_i, j = t mod L_i
      zig-zag:    chunk c = t div C_i (C_i = S_i / 2N); c < N: d = c, j = t mod C_i;
                  else d = 2N-1-c, j = C_i + t mod C_i.
    The oracle's pos[row] must invert it."""
    if layout == ZIGZAG and any((b - a) % (2 * N) for a, b in zip(cu, cu[1:])):
        pytest.skip("zig-zag needs every length a multiple of 2N")
    S = cu[-1]
    L = S // N
    row_of = {}
    for i in range(len(cu) - 1):
        Si = cu[i + 1] - cu[i]
        Li = Si // N
        for t in range(Si):
            if layout == STRIPED:
                d, j = t % N, t // N
            elif layout == CONTIGUOUS:
                d, j = t // Li, t % Li
            else:
                Ci = Si // (2 * N)
                c = t // Ci
                d, j = (c, t % Ci) if c < N else (2 * N - 1 - c, Ci + t % Ci)
            row_of[cu[i] + t] = d * L + cu[i] // N + j
    assert sorted(row_of.values()) == list(range(S))
    pos = oracle.varlen_positions(cu, N, layout)
    for p, row in row_of.items():
        assert pos[row] == p, (p, row)


@pytest.mark.parametrize("layout", [STRIPED, CONTIGUOUS, ZIGZAG])
def test_bwd_block_rounds_sum_to_the_full_backward(oracle_lib, layout):
    """The per-round gradient shares of every (device, key block) pair of the
    ring add up to the full backward (pinned itself to torch autograd): dq
    of a query row over its device's N rounds, dk / dv of a key row over the
    N devices that see its block."""
    S, D, N = 64, 8, 4
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((S, D)) for _ in range(4))
    scale = 0.4
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(q, k, v, do, scale)
    lse, J, _ = oracle.bwd_rows(q, k, v, do, scale, want_dq=False)
    pos = oracle.layout_positions(S, N, layout)
    L = S // N
    dq = np.zeros((S, D))
    dk = np.zeros((S, D))
    dv = np.zeros((S, D))
    for d in range(N):
        qp = pos[d * L:(d + 1) * L]
        for r in range(N):
            e = (d - r) % N
            kp = pos[e * L:(e + 1) * L]
            gq, gk, gv = oracle.bwd_block(q[qp], do[qp], qp, lse[qp], J[qp], k[kp], v[kp], kp, scale)
            dq[qp] += gq
            dk[kp] += gk
            dv[kp] += gv
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert np.abs(got - ref).max() < 1e-11


def test_bwd_block_special_cases(oracle_lib):
    """One block holding the whole sequence is the full backward; a block
    whose keys all come after its queries contributes nothing; J_p may be
    taken as <dO_p, O_p> (the distributed form) with the same result."""
    S, D = 24, 6
    rng = np.random.default_rng(6)
    q, k, v, do = (rng.standard_normal((S, D)) for _ in range(4))
    scale = 0.5
    ref = oracle.attn_bwd(q, k, v, do, scale)
    o, lse = oracle.attn_fwd(q, k, v, scale)
    J_dot = np.einsum("pd,pd->p", do, o)
    allpos = np.arange(S)
    got = oracle.bwd_block(q, do, allpos, lse, J_dot, k, v, allpos, scale)
    for g, r in zip(got, ref):
        assert np.abs(g - r).max() < 1e-11
    z = oracle.bwd_block(q[:8], do[:8], allpos[:8], lse[:8], J_dot[:8], k[8:], v[8:], allpos[8:], scale)
    assert all(np.all(x == 0.0) for x in z)
