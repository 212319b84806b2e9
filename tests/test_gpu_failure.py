"""Failure detection on the GPU without a fault: a tensor-core kernel whose
barrier waits cannot be satisfied (its first loads withheld by the test hook)
gives up after its bounded wait, drains, frees its tensor memory and reports
MEDUSA_DEV_TIMEOUT; the context stays usable and the next call is exact."""
import time

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.helpers import TOL, bf16_to_f64, rel_err, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    return m


def test_linear_bounded_wait_reports_timeout_and_context_survives(mg):
    T, K, N = 64, 256, 256  # two CTAs with one whole tile each, fewer K blocks than ring stages
    rng = np.random.default_rng(3)
    x = wl.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    w = wl.to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    dx, dw = to_dev(x), to_dev(w)
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    mg.medusa_linear_test_stall(dx, dw, y, st)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert mg.medusa_status_check(st) == 3  # MEDUSA_DEV_TIMEOUT
    assert 0.5 < waited < 10.0  # the one-second bounded wait, not a hang
    # tensor memory was freed and the context is intact: a normal call is exact
    y2 = mg.medusa_linear(dx, dw, d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    assert rel_err(bf16_to_f64(to_host(y2)), oracle.linear(x, w)) <= TOL["bf16"]
