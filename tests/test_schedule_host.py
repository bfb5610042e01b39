"""The attention kernels' tile schedule, checked on the CPU against the
oracle's causal mask.  `tests/schedule_harness.cu` (host code built from the
kernels' own header) prints, for every (device d, key stripe e), the forward
span of each query tile (fully kept key tiles, the diagonal tile and its
mask offset) and the backward span of each key tile (first query tile, the
diagonal one and its offset).  Every 2-D tile, ragged edges included, must
then hold exactly the pairs the oracle keeps on that placement's positions:
key position <= query position."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import sequence_parallelism_striped_gb300 as sp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    # (layout, S, N, T)
    (sp.STRIPED, 256, 4, 16), (sp.STRIPED, 1200, 4, 128), (sp.STRIPED, 1028, 4, 128),
    (sp.STRIPED, 96, 8, 3), (sp.STRIPED, 90, 3, 4), (sp.STRIPED, 40, 8, 1), (sp.STRIPED, 48, 16, 128),
    (sp.STRIPED, 8192, 8, 128),
    (sp.CONTIGUOUS, 256, 4, 16), (sp.CONTIGUOUS, 1200, 4, 128), (sp.CONTIGUOUS, 1028, 4, 128),
    (sp.CONTIGUOUS, 96, 8, 3), (sp.CONTIGUOUS, 90, 3, 4), (sp.CONTIGUOUS, 40, 8, 1),
    (sp.ZIGZAG, 256, 4, 16), (sp.ZIGZAG, 1536, 12, 64), (sp.ZIGZAG, 96, 2, 8), (sp.ZIGZAG, 2048, 4, 128),
    (sp.ZIGZAG, 64, 4, 1),
]


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("schedule") / "schedule_harness")
    cmd = [nvcc, "-O1", "-std=c++17", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "sequence_parallelism_striped_gb300", "csrc"),
           "-gencode", "arch=compute_103a,code=sm_103a",
           os.path.join(ROOT, "tests", "schedule_harness.cu"), "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def _spans(exe, layout, S, N, T):
    out = subprocess.run([exe, str(layout), str(S), str(N), str(T)], capture_output=True, text=True,
                         check=True).stdout.split("\n")
    fwd, bwd = {}, {}
    for line in out:
        if not line:
            continue
        tag, *v = line.split()
        d, e, t, lo, diag, off = map(int, v)
        (fwd if tag == "R" else bwd)[(d, e, t)] = (lo, diag, off)
    return fwd, bwd


def _expected_tile(rows, cols, kind, off):
    """'all', 'none' or 'diag' (keep local key column <= local query row + off)."""
    if kind == "all":
        return np.ones((rows, cols), dtype=bool)
    if kind == "none":
        return np.zeros((rows, cols), dtype=bool)
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    return c <= r + off


@pytest.mark.parametrize("layout,S,N,T", CASES)
def test_kernel_tile_schedule_equals_oracle_mask(harness, layout, S, N, T):
    L = S // N
    n = -(-L // T)
    pos = oracle.layout_positions(S, N, layout)
    fwd, bwd = _spans(harness, layout, S, N, T)
    assert len(fwd) == len(bwd) == N * N * n
    for d in range(N):
        qpos = pos[d * L:(d + 1) * L]
        for e in range(N):
            kpos = pos[e * L:(e + 1) * L]
            kept = kpos[None, :] <= qpos[:, None]  # [query row, key row] of this stripe pair
            for a in range(n):
                nfull, diag, off = fwd[(d, e, a)]
                for b in range(n):
                    tile = kept[a * T:(a + 1) * T, b * T:(b + 1) * T]
                    kind = "all" if b < nfull else ("diag" if diag and b == nfull else "none")
                    assert np.array_equal(tile, _expected_tile(*tile.shape, kind, off)), (d, e, a, b)
            for b in range(n):
                a_lo, diag, off = bwd[(d, e, b)]
                for a in range(n):
                    tile = kept[a * T:(a + 1) * T, b * T:(b + 1) * T]
                    if a < a_lo:
                        kind = "none"
                    elif a == a_lo and diag:
                        kind = "diag"
                    else:
                        kind = "all"
                    assert np.array_equal(tile, _expected_tile(*tile.shape, kind, off)), (d, e, a, b)


def test_pair_schedule_shares_key_tiles():
    """The stripe-pair forward runs query tile a of stripes d and d + 1 on one
    K/V stream: on whole-tile stripes both visit key tiles 0..a of every key
    stripe, and only the diagonal offset may differ."""
    S, N, T = 4096, 8, 128
    L = S // N
    n = L // T
    pos = oracle.stripe_positions(S, N)
    for d in range(0, N, 2):
        for e in range(N):
            for a in range(n):
                sets = []
                for x in (d, d + 1):
                    q = pos[x * L + a * T:x * L + (a + 1) * T]
                    k = pos[e * L:(e + 1) * L]
                    kept = k[None, :] <= q[:, None]
                    sets.append(np.flatnonzero(kept.reshape(T, n, T).any(axis=(0, 2))))
                assert np.array_equal(sets[0], np.arange(a + 1)) and np.array_equal(sets[1], np.arange(a + 1))
