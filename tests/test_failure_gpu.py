"""The error path of the tensor-core kernels' bounded waits, exercised without a
fault: a wait on a barrier that nothing arrives at runs out, the kernel records
its code in the device error word and returns; the device stays usable (a
library call afterwards still matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B

pytestmark = pytest.mark.gpu


def _topk_still_matches_the_oracle():
    n_cap, k, n_win, m = 256, 16, 128, 4
    p = B.make_params(1, 1, 64, n_win, m, k, 1, 8, B.F32, B.ELIG_DISJOINT, 0.0)
    g = torch.Generator().manual_seed(3)
    scores = torch.randn((1, 1, n_cap), generator=g, dtype=torch.float32)
    t = n_win + m * n_cap - 1                      # every entry eligible
    q_pos = torch.tensor([[t]], dtype=torch.int32, device="cuda")
    idx = torch.full((1, 1, k), -7, dtype=torch.int32, device="cuda")
    B.csa_topk(p, scores.cuda(), n_cap, q_pos, 1, idx)
    torch.cuda.synchronize()
    want = O.topk_select(scores[0, 0].double().numpy(), k)
    np.testing.assert_array_equal(idx[0, 0].cpu().numpy(), want)


def test_a_wait_that_runs_out_records_its_code_and_the_device_stays_usable():
    torch.cuda.init()
    B.ha_device_error(clear=True)
    try:
        _run()
    finally:
        torch.cuda.synchronize()
        B.ha_device_error(clear=True)             # later tests start with no code set


def _run():
    t0 = time.perf_counter()
    B.ha_selftest_wait_timeout(77)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert B.ha_device_error(clear=False) == 77
    assert 1.5 < waited < 60, waited                # the 2 s limit, not an early exit
    # the first code wins: a second wait that runs out leaves it in place, and
    # with a code set it gives up at once
    t0 = time.perf_counter()
    B.ha_selftest_wait_timeout(78)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.5          # well under the 2 s limit
    assert B.ha_device_error(clear=True) == 77
    assert B.ha_device_error(clear=False) == 0
    _topk_still_matches_the_oracle()
    assert B.ha_device_error(clear=False) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("wc", [False, True])
def test_host_buffers_are_page_locked_and_round_trip(wc):
    """ha_host_alloc memory as CPU tensors: recognised as pinned, copied to the
    device and back unchanged (write-combined only for host-written inputs)."""
    import torch
    from long_context_hybrid_02_b300 import binding as B
    h = B.host_empty((3, 1000), torch.bfloat16, write_combined=wc)
    assert h.is_pinned() and h.shape == (3, 1000) and h.dtype == torch.bfloat16
    src = torch.randn(3, 1000).to(torch.bfloat16)
    h.copy_(src)
    d = torch.empty((3, 1000), dtype=torch.bfloat16, device="cuda")
    d.copy_(h, non_blocking=True)
    back = B.host_empty((3, 1000), torch.bfloat16)
    back.copy_(d, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
