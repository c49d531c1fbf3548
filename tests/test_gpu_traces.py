"""GPU parity over the PersistentKV trace families.

The summary evaluates Uniform, Bimodal, Zipf-like and Bucketed traces at
batch sizes 1, 4 and 8 ("PersistentKV" gist.science summary, Methodology
section 3 "Evaluation Protocol" and Results).  Each family's batch is drawn by
workloads.trace (its readings of the unpublished parameters are stated there)
and decoded on the policy's own route and on each split route; every result
must match the fp64 oracle within 2e-3 on out and 1e-4 on LSE, with the work
tiles bit-exact against the oracle's enumeration and a clean status word.
"""
import functools

import numpy as np
import pytest
import torch

from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import assert_close, expected_queue, oracle_result, run, to_device

pytestmark = pytest.mark.gpu

ROUTES = ["auto", "split_queue", "split_padded", "persistent"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


@functools.lru_cache(maxsize=1)
def _case(kind, B):
    p = wl.trace(kind, B)
    return p, oracle_result(p, nthreads=16)


@pytest.mark.parametrize("B", [1, 4, 8])
@pytest.mark.parametrize("kind", wl.TRACE_KINDS)
def test_trace_family_every_route(kind, B):
    p, ref = _case(kind, B)
    dev = to_device(p)
    for route in ROUTES:
        opts = {} if route == "auto" else dict(force_mode=route)
        out, lse, plan, _ = run(p, dev=dev, **opts)
        assert_close(out, lse, *ref, what=f"{p.name} {route}")
        info = plan.info()
        if route != "auto":
            assert info["mode_name"] == route
        assert np.array_equal(plan.queue(), expected_queue(p, info)), f"{p.name} {route}: queue"
        assert plan.status() == 0, f"{p.name} {route}: status"
        plan.close()
        dev["out"].fill_(float("nan"))
        dev["lse"].fill_(float("nan"))
    del dev
    torch.cuda.empty_cache()
