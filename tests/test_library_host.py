"""Host-side checks of libstriped (no GPU needed): the library builds,
loads and exports every entry point of include/striped.h; the exact
per-round tile table and critical path agree with the oracle's brute force
and with the golden tables; argument validation rejects bad input before
touching the device."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle
import sequence_parallelism_striped_gb300 as sp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return sp.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "striped.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "striped_attn_fwd" in names and "ring_round_fwd" in names
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS])
@pytest.mark.parametrize("S,N,Tq,Tk", [(256, 4, 16, 16), (1200, 4, 128, 128), (1028, 4, 128, 128),
                                       (96, 8, 3, 3), (90, 3, 4, 7), (40, 8, 1, 1), (8192, 8, 128, 128),
                                       (64, 1, 16, 16), (4, 4, 128, 128)])
def test_tile_counts_match_oracle_bruteforce(lib, S, N, Tq, Tk, layout):
    full, part = sp.tile_counts(S, N, Tq, Tk, layout)
    bf, bp = oracle.tile_counts_bruteforce(S, N, Tq, Tk, layout)
    assert np.array_equal(full, bf) and np.array_equal(part, bp)
    assert sp.critical_path(S, N, Tq, Tk, layout) == oracle.critical_path(bf, bp)


@pytest.mark.parametrize("S,N,Tq,Tk", [(256, 4, 16, 16), (1024, 4, 128, 128), (1200, 4, 128, 128),
                                       (96, 8, 3, 3), (90, 3, 4, 7), (48, 8, 1, 1), (8192, 8, 128, 128),
                                       (64, 1, 16, 16), (8, 4, 128, 128), (1536, 12, 64, 32)])
def test_zigzag_tile_counts_match_oracle_bruteforce(lib, S, N, Tq, Tk):
    """Zig-zag placement, including tiles that straddle the chunk boundary
    (C not a multiple of T) and Tq != Tk."""
    full, part = sp.tile_counts(S, N, Tq, Tk, sp.ZIGZAG)
    bf, bp = oracle.tile_counts_bruteforce(S, N, Tq, Tk, oracle.ZIGZAG)
    assert np.array_equal(full, bf) and np.array_equal(part, bp)
    assert sp.critical_path(S, N, Tq, Tk, sp.ZIGZAG) == oracle.critical_path(bf, bp)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
@pytest.mark.parametrize("N,cu,T", [(4, [0, 64, 192, 256], 16), (8, [0, 1024, 3072, 8192], 128),
                                    (4, [0, 40, 48, 88], 4), (2, [0, 8, 12, 20, 32], 3)])
def test_varlen_tile_counts_match_oracle(lib, N, cu, T, layout):
    """Packed batch: the sum of the oracle's brute-force tables of the
    sequences; the critical path takes the busiest device of that sum (not
    the sum of the sequences' critical paths)."""
    if layout == sp.ZIGZAG and any((b - a) % (2 * N) for a, b in zip(cu, cu[1:])):
        pytest.skip("zig-zag needs every length a multiple of 2N")
    full, part = sp.tile_counts_varlen(cu, N, T, T, layout)
    bf = sum(oracle.tile_counts_bruteforce(b - a, N, T, T, layout)[0] for a, b in zip(cu, cu[1:]))
    bp = sum(oracle.tile_counts_bruteforce(b - a, N, T, T, layout)[1] for a, b in zip(cu, cu[1:]))
    assert np.array_equal(full, bf) and np.array_equal(part, bp)
    assert sp.critical_path_varlen(cu, N, T, T, layout) == oracle.critical_path(bf, bp)


def test_varlen_contiguous_critical_path_exceeds_striped(lib):
    """Packing does not fix Ring Attention's imbalance: with several long
    sequences the contiguous placement's critical path stays far above the
    striped one."""
    cu, N, T = [0, 8192, 16384, 24576, 32768], 8, 128
    cs = sp.critical_path_varlen(cu, N, T, T, sp.STRIPED)
    cc = sp.critical_path_varlen(cu, N, T, T, sp.CONTIGUOUS)
    assert cc > 1.6 * cs


def test_golden_tables(lib):
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "tile_counts.json")))
    for w in gold["workloads"]:
        S, N, T = w["S"], w["N"], w["T"]
        for name, layout in (("striped", sp.STRIPED), ("contiguous", sp.CONTIGUOUS), ("zigzag", sp.ZIGZAG)):
            full, part = sp.tile_counts(S, N, T, T, layout)
            assert full.tolist() == w[name]["full"], (w["name"], name)
            assert part.tolist() == w[name]["partial"], (w["name"], name)
            assert sp.critical_path(S, N, T, T, layout) == w[name]["critical_path"]


def test_kernel_tiles(lib):
    import torch

    assert sp.kernel_tile(torch.bfloat16, 128) == 128
    assert sp.kernel_tile(torch.bfloat16, 64) == 128
    assert sp.kernel_tile(torch.float32, 64) == 16
    with pytest.raises(sp.StripedError):
        sp.kernel_tile(torch.bfloat16, 96)


def test_forward_schedule_rule(lib):
    """Stripe-pair forward (2 query tiles per CTA) only for bf16, D = 64 or 128,
    striped, whole-tile stripes, even N, and a balanced grid: twice the
    heaviest pair CTA's key tiles (2 * nq * N) at most the average key
    tiles per multiprocessor, the total taken from the oracle's table."""
    import torch

    sms = 152
    cases = [(1, 32, 262144, 8), (1, 8, 65536, 8), (1, 8, 8192, 8), (1, 24, 8192, 8), (2, 24, 4096, 2),
             (1, 24, 6144, 6), (1, 8, 16384, 8), (1, 8, 32768, 8), (4, 32, 2048, 8), (1, 2, 1536, 3),
             (1, 2, 1200, 4), (1, 64, 1024, 4)]
    seen = set()
    for B, H, S, N in cases:
        L = S // N
        full, part = oracle.tile_counts_closed(S, N, 128, sp.STRIPED) if L % 128 == 0 else (None, None)
        if L % 128 == 0 and N % 2 == 0:
            total = B * H * int(full.sum() + part.sum())
            heaviest = 2 * (L // 128) * N
            want = 2 if 2 * heaviest * sms <= total else 1
        else:
            want = 1
        got = sp.fwd_query_tiles_per_cta(B, H, S, 128, N, sp.STRIPED, torch.bfloat16, num_sms=sms)
        assert got == want, (B, H, S, N)
        seen.add(got)
    assert seen == {1, 2}
    # the benchmark sizes take the pair schedule, the short-sequence one does not
    assert sp.fwd_query_tiles_per_cta(1, 32, 262144, 128, 8, num_sms=sms) == 2
    assert sp.fwd_query_tiles_per_cta(1, 8, 8192, 128, 8, num_sms=sms) == 1
    # every other kernel configuration: one query tile per CTA
    for layout in (sp.CONTIGUOUS, sp.ZIGZAG):
        assert sp.fwd_query_tiles_per_cta(1, 32, 262144, 128, 8, layout, num_sms=sms) == 1
    # head dimension 64 follows the same rule as 128
    assert sp.fwd_query_tiles_per_cta(1, 32, 262144, 64, 8, num_sms=sms) == 2
    assert sp.fwd_query_tiles_per_cta(1, 8, 8192, 64, 8, num_sms=sms) == 1
    assert sp.fwd_query_tiles_per_cta(1, 4, 4096, 64, 8, dtype=torch.float32, num_sms=sms) == 1
    # more multiprocessors need more work per head before pairs pay
    assert sp.fwd_query_tiles_per_cta(1, 24, 8192, 128, 8, num_sms=1000) == 1
    for bad in ((1, 32, 262144, 96, 8, sp.STRIPED, torch.bfloat16, sms),
                (1, 32, 262144, 128, 8, sp.STRIPED, torch.bfloat16, 0),
                (1, 32, 262144, 128, 8, 7, torch.bfloat16, sms),
                (1, 32, 262143, 128, 8, sp.STRIPED, torch.bfloat16, sms)):
        with pytest.raises(sp.StripedError):
            sp.fwd_query_tiles_per_cta(*bad[:5], bad[5], bad[6], num_sms=bad[7])


def test_invalid_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    # NULL pointers
    assert lib.striped_attn_fwd(None, fake, fake, fake, fake, 1, 1, 64, 128, 4, 0, 0, 1.0, None, None) == -1
    # S % N != 0
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 66, 128, 4, 0, 0, 1.0, None, None) == -1
    # unsupported head dim for bf16
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 64, 96, 4, 0, 0, 1.0, None, None) == -2
    # bad layout / dtype
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 64, 128, 4, 7, 0, 1.0, None, None) == -1
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 64, 128, 4, 0, 9, 1.0, None, None) == -1
    # misaligned pointer
    assert lib.striped_attn_fwd(P((1 << 20) + 2), fake, fake, fake, fake, 1, 1, 64, 128, 4, 0, 0, 1.0, None,
                                None) == -3
    # permute: overlapping buffers, bad sizes
    assert lib.striped_permute(fake, fake, 1, 1, 64, 128, 4, 0, None) == -1
    assert lib.striped_permute(fake, P((1 << 24)), 1, 1, 64, 128, 0, 0, None) == -1
    # permute: a row must be whole 16-byte vectors (bf16 D = 12: 24 bytes), at most 32 KB
    # (fp32 D = 16384: 64 KB); any vector count in between is taken
    assert lib.striped_permute(fake, P((1 << 24)), 1, 1, 64, 12, 4, 0, None) == -3
    assert lib.striped_permute(fake, P((1 << 24)), 1, 1, 64, 16384, 4, 1, None) == -2
    # workspace too small
    assert lib.striped_attn_bwd(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 16, 1, 1, 64, 128,
                                4, 0, 0, 1.0, None, None) == -6
    # ring round: bad device index
    assert lib.ring_round_fwd(fake, fake, fake, fake, fake, None, 5, 0, 1, 1, 16, 128, 4, 16 * 128, 16, 0, 0,
                              1.0, 1, None, None) == -1
    assert lib.striped_tile_counts(65, 4, 16, 16, 0, None, None) == -1
    assert lib.striped_critical_path(64, 0, 16, 16, 0) < 0
    # zig-zag: S must split into 2N chunks; chunks must be whole kernel tiles
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 1028, 128, 4, 2, 0, 1.0, None, None) == -1
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 1200, 128, 4, 2, 0, 1.0, None, None) == -2
    assert lib.striped_attn_fwd(fake, fake, fake, fake, fake, 1, 1, 200, 64, 4, 2, 1, 1.0, None, None) == -2
    assert lib.striped_layout_permute(fake, P(1 << 24), 1, 1, 12, 128, 4, 2, 0, None) == -1
    assert lib.striped_layout_permute(fake, P(1 << 24), 1, 1, 16, 128, 4, 3, 0, None) == -1
    assert lib.striped_tile_counts(36, 4, 16, 16, 2, None, None) == -1
    # grouped-query attention: Hkv must divide H
    assert lib.striped_attn_fwd_gqa(fake, fake, fake, fake, fake, 1, 6, 4, 64, 128, 4, 0, 0, 1.0, None,
                                    None) == -1
    assert lib.striped_attn_fwd_gqa(fake, fake, fake, fake, fake, 1, 4, 0, 64, 128, 4, 0, 0, 1.0, None,
                                    None) == -1
    assert lib.striped_attn_bwd_gqa(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30, 1, 4, 8,
                                    64, 128, 4, 0, 0, 1.0, None, None) == -1
    # packed sequences: cu_seqlens checked on the host
    def cu(vals):
        arr = (ctypes.c_int32 * len(vals))(*vals)
        return arr, len(vals) - 1

    def fwd_varlen(vals, N=4, layout=0, dtype=0):
        arr, n = cu(vals)
        return lib.striped_attn_fwd_varlen(fake, fake, fake, fake, fake, arr, n, 2, 2, 128, N, layout, dtype, 1.0,
                                           None, None)

    assert fwd_varlen([1, 512, 1024]) == -1           # does not start at 0
    assert fwd_varlen([0, 1024, 512]) == -1           # decreasing
    assert fwd_varlen([0, 512, 514]) == -1            # length not a multiple of N
    assert fwd_varlen([0, 512, 516]) == -2            # multiple of N, not of N*T
    assert fwd_varlen([0, 512, 1024], layout=2) == -2  # zig-zag: 512 is not a multiple of 2N*T
    assert fwd_varlen([0, 512, 1028], layout=2) == -1  # zig-zag: not a multiple of 2N
    assert fwd_varlen(list(range(0, 513 * 512 + 1, 512))) == -2  # more than 512 sequences
    arr, n = cu([0, 6, 12])
    assert lib.striped_varlen_permute(fake, P(1 << 24), arr, n, 1, 64, 4, 2, 0, None) == -1
    # NULL table, NULL tensors, misaligned tensors, bad head dimension
    assert lib.striped_attn_fwd_varlen(fake, fake, fake, fake, fake, None, 2, 2, 2, 128, 4, 0, 0, 1.0, None,
                                       None) == -1
    arr, n = cu([0, 512, 1024])
    assert lib.striped_attn_fwd_varlen(None, fake, fake, fake, fake, arr, n, 2, 2, 128, 4, 0, 0, 1.0, None,
                                       None) == -1
    assert lib.striped_attn_fwd_varlen(P((1 << 20) + 8), fake, fake, fake, fake, arr, n, 2, 2, 128, 4, 0, 0,
                                       1.0, None, None) == -3
    assert lib.striped_attn_fwd_varlen(fake, fake, fake, fake, fake, arr, n, 2, 2, 96, 4, 0, 0, 1.0, None,
                                       None) == -2
    assert lib.striped_attn_bwd_varlen(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 16, arr, n, 2,
                                       2, 128, 4, 0, 0, 1.0, None, None) == -6  # workspace too small
    assert lib.striped_tile_counts_varlen(None, 2, 4, 16, 16, 0, None, None) == -1
    assert lib.striped_critical_path_varlen(arr, n, 0, 16, 16, 0) < 0
    # grouped-query: misaligned key/value tensor
    assert lib.striped_attn_fwd_gqa(fake, P((1 << 20) + 4), fake, fake, fake, 1, 4, 2, 64, 128, 4, 0, 0, 1.0,
                                    None, None) == -3
    # bf16 head dimension 64 accepted by validation (fails later only on a NULL output)
    assert lib.striped_attn_fwd(fake, fake, fake, None, fake, 1, 1, 64, 64, 4, 0, 0, 1.0, None, None) == -1


def test_workspace_size(lib):
    import torch

    B, H, S, D, N = 2, 3, 512, 128, 4
    n = sp.workspace_size(B, H, S, D, N, torch.bfloat16)
    assert n >= B * H * S * D * 4 + 2 * B * H * S * 4 and n % 256 == 0
    # statistics are padded to whole 128-row tiles per stripe: L = 129 -> 2 tiles
    assert sp.workspace_size(1, 1, 4 * 129, D, 4, torch.bfloat16) >= 4 * 129 * D * 4 + 4 * 2 * 256 * 4
    assert sp.workspace_size(1, 1, 256, 64, 4, torch.float32) >= 256 * 4
    assert sp.workspace_size(1, 1, 257, 64, 4, torch.float32) == 0


def test_status_strings(lib):
    assert sp.status_string(0) == "ok"
    assert "timed out" in sp.status_string(-5)


def test_test_hook_rejects_unknown_faults(lib):
    """The fault-injection test hook validates its selector before it
    touches the device."""
    assert lib.striped_test_inject(3, 0) == -1
    assert lib.striped_test_inject(-1, 1000) == -1
    assert "striped_test_inject" in _declared_functions()

