"""Stripe permutation on the GPU: bit-exact against the placement the oracle
builds by enumeration ("every N-th token"; for the zig-zag placement, chunks
d and 2N-1-d), and round trip."""
import pytest
import torch

import oracle
import sequence_parallelism_striped_gb300 as sp
from tests._util import positions

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 1, 256, 64, 4), (2, 3, 1200, 128, 4), (1, 8, 8192, 128, 8),
                                       (1, 2, 4096, 64, 16), (1, 1, 40, 128, 8), (1, 2, 384, 128, 1),
                                       (1, 1, 48, 32, 48)])
def test_permute_bit_exact(B, H, S, D, N, dtype):
    dev = torch.device("cuda")
    g = torch.Generator(device="cpu").manual_seed(123)
    x = torch.randn(B, H, S, D, generator=g).to(dtype)
    pos = torch.as_tensor(positions(S, N, sp.STRIPED))
    ref = x[:, :, pos]  # row r holds position pos[r]
    y = sp.striped_permute(x.to(dev), N)
    assert torch.equal(y.cpu(), ref)
    z = sp.striped_unpermute(y, N)
    assert torch.equal(z.cpu(), x)


@pytest.mark.parametrize("layout", [sp.STRIPED, sp.CONTIGUOUS, sp.ZIGZAG])
@pytest.mark.parametrize("B,H,S,D,N,dtype", [
    (1, 2, 6 * 38, 96, 6, torch.float32),   # rows of 24 16-byte vectors (not a power of two)
    (2, 1, 10 * 20, 24, 5, torch.bfloat16),  # rows of 3 vectors
    (1, 1, 8 * 64, 96, 8, torch.bfloat16),   # rows of 12 vectors
])
def test_permute_rows_not_a_power_of_two(B, H, S, D, N, dtype, layout):
    """Row sizes that are not a power of two of 16-byte vectors (the fp32
    attention path accepts any head dimension that is a multiple of 8) take
    the permutation's division path: bit-exact and a round trip."""
    dev = torch.device("cuda")
    g = torch.Generator(device="cpu").manual_seed(77)
    x = torch.randn(B, H, S, D, generator=g).to(dtype)
    pos = torch.as_tensor(positions(S, N, layout))
    y = sp.layout_permute(x.to(dev), N, layout)
    assert torch.equal(y.cpu(), x[:, :, pos])
    assert torch.equal(sp.layout_unpermute(y, N, layout).cpu(), x)


def test_permute_full_size_long_context():
    """Largest tensor of the benchmark workloads (B=1, H=32, S=262144,
    D=128, bf16, N=8): sampled rows bit-exact, round trip exact."""
    dev = torch.device("cuda")
    B, H, S, D, N = 1, 32, 262144, 128, 8
    g = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn(B, H, S, D, generator=g, device=dev).to(torch.bfloat16)
    y = sp.striped_permute(x, N)
    L = S // N
    rows = torch.randint(0, S, (4096,), generator=torch.Generator().manual_seed(9))
    heads = torch.randint(0, H, (4096,), generator=torch.Generator().manual_seed(10))
    d, i = rows // L, rows % L
    got = y[0, heads.to(dev), rows.to(dev)]
    want = x[0, heads.to(dev), (i * N + d).to(dev)]
    assert torch.equal(got, want)
    assert torch.equal(sp.striped_unpermute(y, N), x)


@pytest.mark.parametrize("layout", [sp.ZIGZAG, sp.CONTIGUOUS, sp.STRIPED])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,S,D,N", [(1, 1, 256, 64, 4), (2, 3, 1200, 128, 4), (1, 8, 8192, 128, 8),
                                       (1, 2, 4096, 64, 16), (1, 1, 48, 128, 8), (1, 2, 384, 128, 1),
                                       (1, 1, 96, 32, 48)])
def test_layout_permute_bit_exact(B, H, S, D, N, dtype, layout):
    dev = torch.device("cuda")
    g = torch.Generator(device="cpu").manual_seed(321)
    x = torch.randn(B, H, S, D, generator=g).to(dtype)
    pos = torch.as_tensor(positions(S, N, layout))
    y = sp.layout_permute(x.to(dev), N, layout)
    assert torch.equal(y.cpu(), x[:, :, pos])
    assert torch.equal(sp.layout_unpermute(y, N, layout).cpu(), x)


def test_zigzag_permute_full_size_long_context():
    """Zig-zag placement of the largest benchmark tensor (B=1, H=32,
    S=262144, D=128, bf16, N=8): sampled rows bit-exact, round trip exact."""
    dev = torch.device("cuda")
    B, H, S, D, N = 1, 32, 262144, 128, 8
    g = torch.Generator(device=dev).manual_seed(6)
    x = torch.randn(B, H, S, D, generator=g, device=dev).to(torch.bfloat16)
    y = sp.layout_permute(x, N, sp.ZIGZAG)
    rows = torch.randint(0, S, (4096,), generator=torch.Generator().manual_seed(11))
    heads = torch.randint(0, H, (4096,), generator=torch.Generator().manual_seed(12))
    pos = torch.as_tensor([int(oracle.position_of_row(int(r), S, N, oracle.ZIGZAG)) for r in rows])
    got = y[0, heads.to(dev), rows.to(dev)]
    want = x[0, heads.to(dev), pos.to(dev)]
    assert torch.equal(got, want)
    assert torch.equal(sp.layout_unpermute(y, N, sp.ZIGZAG), x)
