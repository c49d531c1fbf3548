"""Failure detection on the GPU without a GPU fault.

The kernels' waits are bounded in time: a wait that runs out sets
PKV_DEV_TIMEOUT in the status word, raises the CTA's abort flag (so later waits
of that CTA return at once) and returns.  The self-test entry point makes one
such wait run out on an mbarrier phase that nothing completes, with a short
limit, and the context must stay usable afterwards.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import assert_close, oracle_result, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def test_wait_that_nothing_completes_times_out_and_reports():
    status, (first_ok, abort_raised, second_ok) = pkv.selftest_wait(50_000_000)   # 50 ms
    assert status & pkv.DEV_TIMEOUT
    assert first_ok == 0 and abort_raised == 1 and second_ok == 0
    # the context is still usable: an ordinary decode runs and matches the oracle
    p = wl.tiny()
    out, lse, plan, _ = run(p, force_mode="split_queue", num_splits=2)
    assert_close(out, lse, *oracle_result(p), what="after the timeout self-test")
    assert plan.status() == 0


def test_selftest_rejects_bad_limits():
    with pytest.raises(pkv.PkvError):
        pkv.selftest_wait(0)
    with pytest.raises(pkv.PkvError):
        pkv.selftest_wait(3_000_000_000)
