"""The per-CTA timeline of the attention launch (pkv_trace_enable / pkv_trace_read).

Each CTA's row must be a consistent timeline (entry, grid dependency wait,
first block, last block, combine, arrival, merge, exit in that order), the
tile counts must add up to the launch's tiles, exactly one CTA per split
(row, KV head) must have merged, and tracing must not change a single output
bit: a traced decode equals an untraced one, which also checks that two runs
of the same decode agree bitwise.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import assert_close, oracle_result, run, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _problem():
    return wl.make_problem("edges", [1, 15, 16, 17, 32, 33, 0, 250, 700], Hq=8, Hkv=2, D=128, page_size=16,
                           num_pages=96, seed=23)


@pytest.mark.parametrize("route", ["direct", "split_queue", "split_padded", "persistent"])
def test_timeline_rows_are_consistent_and_change_nothing(route):
    p = _problem()
    ref = oracle_result(p)
    dev = to_device(p)
    out0, lse0, plan, _ = run(p, dev=dev, force_mode=route, num_splits=3)
    out0, lse0 = out0.copy(), lse0.copy()
    out1, lse1, _, _ = run(p, dev=dev, plan=plan)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1), "two runs differ"
    plan.trace(True)
    out2, lse2, _, _ = run(p, dev=dev, plan=plan)
    rows = plan.read_trace()
    plan.trace(False)
    assert np.array_equal(out0, out2) and np.array_equal(lse0, lse2), "tracing changed the result"
    assert_close(out2, lse2, *ref, what=route)
    assert plan.status() == 0

    info = plan.info()
    assert rows.shape == (info["grid_ctas"], pkv.TRACE_WORDS)
    num_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert np.all(rows[:, pkv.TR_SM] < num_sms)
    tiles = rows[:, pkv.TR_TILES].astype(np.int64)
    expect_tiles = {"direct": p.B * p.Hkv, "split_padded": info["num_tiles"]}.get(route, info["num_work_items"])
    assert tiles.sum() == expect_tiles
    t = rows.astype(np.int64)
    assert np.all(t[:, pkv.TR_ENTRY] > 0) and np.all(t[:, pkv.TR_ENTRY] <= t[:, pkv.TR_WAIT_DONE])
    assert np.all(t[:, pkv.TR_WAIT_DONE] <= t[:, pkv.TR_EXIT])
    ran = tiles > 0
    streamed = ran & (t[:, pkv.TR_FIRST_BLOCK] > 0)
    for a, b in ((pkv.TR_WAIT_DONE, pkv.TR_FIRST_BLOCK), (pkv.TR_FIRST_BLOCK, pkv.TR_STREAM_END)):
        assert np.all(t[streamed, a] <= t[streamed, b]), (a, b)
    for a, b in ((pkv.TR_STREAM_END, pkv.TR_COMBINE_END), (pkv.TR_COMBINE_END, pkv.TR_EXIT)):
        assert np.all(t[ran, a] <= t[ran, b]), (a, b)
    merged = t[:, pkv.TR_MERGE_END] > 0
    arrived = t[:, pkv.TR_ARRIVED] > 0
    assert np.all(t[merged, pkv.TR_ARRIVED] > 0)
    assert np.all(t[arrived, pkv.TR_ARRIVED] <= t[arrived, pkv.TR_EXIT])
    assert np.all(t[merged, pkv.TR_MERGE_END] <= t[merged, pkv.TR_EXIT])
    # (row, KV head) units whose split tiles are merged: every unit of the padded
    # grid, the units with more than one tile in the compact queue
    q = plan.queue()
    split_units = {(int(b), int(h)) for b, h, s, _, _ in q if s > 0}
    if route == "direct":
        assert not merged.any() and not arrived.any()
    elif route == "persistent":   # a CTA may merge for one tile and then run others
        assert 1 <= merged.sum() <= len(split_units)
    else:                         # one tile per CTA: exactly one merging CTA per split unit
        assert np.all(t[merged, pkv.TR_ARRIVED] <= t[merged, pkv.TR_MERGE_END])
        assert merged.sum() == len(split_units)
        got = {(int(x >> 40), int((x >> 20) & 0xFFFFF)) for x in rows[merged, pkv.TR_LAST_TILE]}
        assert got == split_units
