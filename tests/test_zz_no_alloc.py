"""striped_attn_bwd_noalloc: the backward for callers that cannot allocate
device memory (their memory belongs to an allocator or budget they cannot
extend, or they keep cudaMalloc off the hot path).  Its scratch is a fixed
array inside the library, so this test calls it through the C ABI and
checks it against striped_attn_bwd with a caller-owned workspace, twice in
a row (the second call must not depend on what the first left in the
shared array).  Both run the same kernels: dK and dV are accumulated in a
fixed order and must be equal bit for bit; dQ is summed with fp32 atomics,
so only its summation order may differ.  Collected last on purpose."""
import ctypes

import pytest
import torch

import sequence_parallelism_striped_gb300 as sp
from tests._util import TOL, inputs, maxerr, to_layout

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _fn(lib):
    f = lib.striped_attn_bwd_noalloc
    P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, I, F, P, P]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype,B,H,S,D,N,layout", [
    (torch.bfloat16, 1, 2, 1200, 128, 4, sp.STRIPED),
    (torch.bfloat16, 1, 8, 8192, 128, 8, sp.STRIPED),
    (torch.bfloat16, 1, 2, 1028, 128, 4, sp.CONTIGUOUS),
    (torch.float32, 1, 1, 256, 64, 4, sp.STRIPED),
])
def test_noalloc_matches_workspace_entry_point(dtype, B, H, S, D, N, layout):
    lib = sp.load()
    fn = _fn(lib)
    x = inputs(B, H, S, D, dtype, seed=11)
    q, k, v, do = (to_layout(x[n], N, layout, DEV) for n in ("q", "k", "v", "do"))
    o, lse = sp.striped_attn_fwd(q, k, v, N, layout)
    scale = 1.0 / D ** 0.5
    ref = sp.striped_attn_bwd(q, k, v, o, lse, do, N, layout, scale=scale)
    code = sp.BF16 if dtype == torch.bfloat16 else sp.FP32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    tol = TOL[dtype]["grad"]
    for _ in range(2):
        dq, dk, dv = (torch.full_like(q, 7.0) for _ in range(3))
        st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                B, H, S, D, N, layout, code, scale, None, stream)
        assert st == 0, sp.status_string(st)
        torch.cuda.synchronize()
        assert sp.check_error() == 0
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert maxerr(dq.float().cpu(), ref[0].float().cpu()) <= tol


def test_noalloc_rejects_problems_beyond_the_array():
    """A problem whose workspace exceeds the fixed array is refused up front
    (no kernel runs, nothing is written)."""
    lib = sp.load()
    fn = _fn(lib)
    fake = ctypes.c_void_p(1 << 20)
    # B=1, H=32, S=262144, D=128 needs ~4.3 GB of scratch
    st = fn(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 32, 262144, 128, 8, sp.STRIPED, sp.BF16,
            0.088, None, None)
    assert st == -6
