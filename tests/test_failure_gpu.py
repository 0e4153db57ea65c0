"""The bounded-wait failure path on the GPU, without any fault: a wait on an
mbarrier that nothing completes runs out after its limit, the kernel raises
the device fault flag and returns, and the host reads TR_ERR_TIMEOUT; the
context stays usable and the flag clears on reading."""
import time

import pytest

from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()
    assert B.tr_device_status() == B.Status.OK


def test_wait_that_completes_reports_ok():
    B.check(B.tr_selftest_bounded_wait(1, 50_000_000))
    assert B.tr_device_status() == B.Status.OK


def test_wait_that_runs_out_reports_timeout_and_clears():
    t0 = time.time()
    B.check(B.tr_selftest_bounded_wait(0, 20_000_000))  # 20 ms
    assert B.tr_device_status() == B.Status.ERR_TIMEOUT
    assert time.time() - t0 < 10
    assert B.tr_device_status() == B.Status.OK  # read clears it


def test_context_still_usable_after_a_timeout():
    import torch
    B.check(B.tr_selftest_bounded_wait(0, 1_000_000))
    assert B.tr_device_status() == B.Status.ERR_TIMEOUT
    x = torch.randn(300, 200, device="cuda")
    assert torch.equal(B.transpose(x, variant=B.Variant.TMA), x.t())
    assert B.tr_device_status() == B.Status.OK


def test_selftest_argument_errors():
    assert B.tr_selftest_bounded_wait(0, 0) == B.Status.ERR_BAD_DIM
    assert B.tr_selftest_bounded_wait(0, 3_000_000_000) == B.Status.ERR_BAD_DIM
