"""Failure detection without a GPU fault: a bounded device wait on a flag
that nothing sets runs out, records a timeout status, and the context stays
usable."""
import pytest
import torch

import sequence_parallelism_striped_gb300 as sp

pytestmark = pytest.mark.gpu


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
