"""pkv_decode_static: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc when they decode: code running inside
another framework's memory budget, real-time loops that must not touch the
allocator, hosts that forbid allocation after start-up.  pkv_decode_static
keeps its split workspace in a fixed device array inside the library instead
of a plan.  These tests call it through the C ABI and compare it with the fp64
oracle on the same inputs, within the tolerances the parity tests use, over
calls in a row with different shapes, so that the shared array's leftover
contents from one call cannot leak into the next.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import assert_close, oracle_result, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _static(p, dev, num_splits, max_seq_len=None):
    out = torch.full_like(dev["out"], float("nan"))
    lse = torch.full_like(dev["lse"], float("nan"))
    pkv.decode_static(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], out, lse,
                      page_size=p.page_size,
                      max_seq_len=int(p.seq_lens.max()) if max_seq_len is None else max_seq_len,
                      num_splits=num_splits, num_pages=p.num_pages)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def test_static_matches_the_oracle_on_calls_in_a_row():
    mixed = wl.mixed()
    edges = wl.make_problem("edges", [1, 15, 16, 17, 0, 250], Hq=8, Hkv=2, D=128, page_size=16,
                            num_pages=40, seed=31)
    dm, de = to_device(mixed), to_device(edges)
    ref_m, ref_e = oracle_result(mixed), oracle_result(edges)
    assert_close(*_static(mixed, dm, 8), *ref_m, what="mixed, first call")
    assert_close(*_static(edges, de, 3), *ref_e, what="edges, second call")   # array holds the first's data
    assert_close(*_static(mixed, dm, 8), *ref_m, what="mixed, third call")


def test_static_poisons_only_rows_beyond_its_split_grid():
    """max_seq_len 100 with 2 splits: P = 7 pages, C = 4, S_max = 2, so rows of up
    to 8 pages (128 tokens) are decoded exactly and the 250-token row (16 pages)
    is poisoned with NaN without reading KV."""
    p = wl.make_problem("over", [100, 250, 128, 0], Hq=8, Hkv=2, D=64, page_size=16, num_pages=40, seed=37)
    dev = to_device(p)
    out, lse = _static(p, dev, 2, max_seq_len=100)
    ref_out, ref_lse = oracle_result(p)
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(lse[1]))
    keep = [0, 2, 3]
    assert_close(out[keep], lse[keep], ref_out[keep], ref_lse[keep], what="rows within the grid")


def test_static_rejects_problems_beyond_its_array():
    """64 rows x 8 KV heads x 64 splits x 4 heads x 129 floats > 8 MiB: PKV_ENOSPACE
    before any launch.  Every buffer has the declared geometry's shape (empty rows,
    tables of -1), so even a launch would read only valid memory."""
    B, Hq, Hkv, D, ps, max_pages, num_pages = 64, 32, 8, 128, 16, 4096, 16
    q = torch.zeros((B, Hq, D), dtype=torch.int16, device="cuda")
    k = torch.zeros((num_pages, ps, Hkv, D), dtype=torch.int16, device="cuda")
    v = torch.zeros_like(k)
    table = torch.full((B, max_pages), -1, dtype=torch.int32, device="cuda")
    lens = torch.zeros((B,), dtype=torch.int32, device="cuda")
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, Hq), dtype=torch.float32, device="cuda")
    geom = pkv.Geom(B, Hq, Hkv, D, max_pages, num_pages)
    rc = pkv.load().pkv_decode_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), table.data_ptr(), lens.data_ptr(),
                                      ps, geom, max_pages * ps, 64, out.data_ptr(), lse.data_ptr(), None)
    assert rc == pkv.ENOSPACE
