"""The bounded waits give up instead of hanging: a device wait on an mbarrier
that nothing arrives on returns after its limit with KVP_ERR_TIMEOUT in the
error word, and the context stays usable; a satisfied wait records nothing."""

import time

import pytest
import torch

from libbuild import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


def test_wait_with_no_arrival_times_out(kb):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kb.kvp_selftest_wait(20_000_000, 0, err)  # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) == kb.KVP_ERR_TIMEOUT
    assert 0.015 <= dt < 1.0, f"the wait took {dt:.3f} s"
    # the context is still usable
    x = torch.arange(1024, device=DEV, dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2


def test_satisfied_wait_records_nothing(kb):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kb.kvp_selftest_wait(20_000_000, 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
