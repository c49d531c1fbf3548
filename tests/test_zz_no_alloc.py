"""pkv_decode_static: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc when they decode: code running inside
another framework's memory budget, real-time loops that must not touch the
allocator, hosts that forbid allocation after start-up.  pkv_decode_static
keeps its split workspace in a fixed device array inside the library instead
of a plan.  These tests call it through the C ABI and compare it with the
planned entry point (pkv_plan + pkv_decode) on the same inputs, within the
tolerances the parity tests use, over two calls in a row so that the shared
array's leftover contents from one call cannot leak into the next.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import LSE_TOL, OUT_TOL, make_plan, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _planned(p, dev, num_splits):
    plan = make_plan(p, force_mode="split_padded", num_splits=num_splits)
    pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
    torch.cuda.synchronize()
    assert plan.status() == 0
    return dev["out"].cpu().numpy().copy(), dev["lse"].cpu().numpy().copy()


def _static(p, dev, num_splits):
    out = torch.full_like(dev["out"], float("nan"))
    lse = torch.full_like(dev["lse"], float("nan"))
    pkv.decode_static(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], out, lse,
                      page_size=p.page_size, max_seq_len=int(p.seq_lens.max()), num_splits=num_splits,
                      num_pages=p.num_pages)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _close(a, b):
    out, lse = a
    ref_out, ref_lse = b
    assert np.all(np.isfinite(out))
    assert np.max(np.abs(out - ref_out)) <= OUT_TOL
    neg = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), neg)
    if np.any(~neg):
        assert np.max(np.abs(lse[~neg] - ref_lse[~neg])) <= LSE_TOL


def test_static_matches_planned_on_two_calls_in_a_row():
    mixed = wl.mixed()
    edges = wl.make_problem("edges", [1, 15, 16, 17, 0, 250], Hq=8, Hkv=2, D=128, page_size=16,
                            num_pages=40, seed=31)
    dm, de = to_device(mixed), to_device(edges)
    ref_m = _planned(mixed, dm, 8)
    ref_e = _planned(edges, de, 3)
    _close(_static(mixed, dm, 8), ref_m)    # first call (sets the array up on this device)
    _close(_static(edges, de, 3), ref_e)    # second call: other shape, array holds the first's data
    _close(_static(mixed, dm, 8), ref_m)    # and back


def test_static_rejects_problems_beyond_its_array():
    p = wl.tiny()
    dev = to_device(p)
    big = pkv.Geom(64, 32, 8, 128, 4096, 1 << 20)   # 64 x 8 x 64 slots of 4 x 129 floats > 8 MiB
    rc = pkv.load().pkv_decode_static(
        dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), dev["table"].data_ptr(),
        dev["lens"].data_ptr(), 16, big, 4096 * 16, 64, dev["out"].data_ptr(), dev["lse"].data_ptr(), None)
    assert rc == pkv.ENOSPACE
