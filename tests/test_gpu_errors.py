"""Failure detection without a GPU fault.

1. A bounded device wait on a flag that nothing sets runs out, records a
   timeout status, and the context stays usable.
2. The attention kernels' own bounded waits: with the test hook the forward
   (or backward) TMA producer never loads its first tile, so every wait on
   that tile runs out after a 1 ms limit.  Each CTA must then record
   STRIPED_ERR_TIMEOUT, wait for its own copies and tensor-core operations
   in flight, free its tensor memory and return; the launch ends, and the
   next normal launch on the same context reproduces the results of a run
   made before the fault (O, LSE, dK, dV bit for bit; dQ up to the order of
   its fp32 atomics).  Nothing faults, traps or hangs: every wait is bounded.
"""
import pytest
import torch

import sequence_parallelism_striped_gb300 as sp
from seeded_inputs import attention_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def test_bounded_wait_reports_timeout():
    torch.cuda.init()
    assert sp.check_error() == 0
    sp.selftest_timeout(10000)
    assert sp.check_error() == -5
    assert sp.check_error() == 0  # cleared by the read
    x = torch.randn(1, 1, 64, 64, device="cuda")
    y = sp.striped_permute(x, 4)
    assert torch.equal(sp.striped_unpermute(y, 4), x)
    assert sp.check_error() == 0


def _run(q, k, v, do, N, layout):
    o, lse = sp.striped_attn_fwd(q, k, v, N, layout)
    dq, dk, dv = sp.striped_attn_bwd(q, k, v, o, lse, do, N, layout)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


# (B, H, S, N, layout, forward query tiles per CTA): the one-tile forward
# (two small heads) and the stripe-pair forward (enough heads to take it)
SHAPES = [(1, 2, 2048, 4, sp.STRIPED, 1), (1, 128, 1024, 4, sp.STRIPED, 2), (1, 2, 2048, 4, sp.CONTIGUOUS, 1)]


@pytest.mark.parametrize("fault", [sp.FAULT_FWD_SKIP_KV, sp.FAULT_BWD_SKIP_Q])
@pytest.mark.parametrize("B,H,S,N,layout,tiles", SHAPES)
def test_kernel_wait_runs_out_and_context_stays_usable(fault, B, H, S, N, layout, tiles):
    D = 128
    assert sp.fwd_query_tiles_per_cta(B, H, S, D, N, layout) == tiles
    x = attention_inputs(B, H, S, D, torch.bfloat16, seed=21)
    q, k, v, do = (sp.layout_permute(x[n].to(DEV), N, layout) for n in ("q", "k", "v", "do"))
    assert sp.check_error() == 0
    ref = _run(q, k, v, do, N, layout)
    assert sp.check_error() == 0
    try:
        sp.test_inject(fault, 1_000_000)  # 1 ms
        o, lse = sp.striped_attn_fwd(q, k, v, N, layout)
        if fault == sp.FAULT_BWD_SKIP_Q:
            # the forward is unaffected; the backward times out
            torch.cuda.synchronize()
            assert sp.check_error() == 0
            sp.striped_attn_bwd(q, k, v, o, lse, do, N, layout)
        assert sp.check_error() == -5
    finally:
        sp.test_inject(sp.FAULT_NONE, 0)
    assert sp.check_error() == 0
    got = _run(q, k, v, do, N, layout)
    assert sp.check_error() == 0
    for name, a, b in zip(("o", "lse", "dk", "dv"), (ref[0], ref[1], ref[3], ref[4]),
                          (got[0], got[1], got[3], got[4])):
        assert torch.equal(a, b), name
    assert (ref[2].float() - got[2].float()).abs().max().item() <= 1e-2
