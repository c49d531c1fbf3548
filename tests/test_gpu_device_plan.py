"""Device-planned continuous steps (pkv_session_device_plan) on the GPU.

The planner kernel must reproduce the host planner bit for bit: page
allocation in row order from the FIFO free list, the queue in (b, kvh, s)
order for the lengths after the append (checked against the oracle's
enumeration), and the longest-first hand-out order (checked against a stable
sort by descending page count).  Outputs are checked against the fp64 oracle,
and a step captured once in a CUDA graph and replayed must give the same
results as eager steps.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from paged_kv_decode_block_gb300.session import ContinuousSessions
from pkv_testutil import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _expected_reserve(lens, table, free, ps):
    for b in range(len(lens)):
        if lens[b] % ps == 0 and table[b, lens[b] // ps] < 0:
            table[b, lens[b] // ps] = free.pop(0)


def _expected_order(queue):
    sizes = queue[:, 4] - queue[:, 3]
    return np.argsort(-sizes, kind="stable").astype(np.int32)


def _ragged_problem(steps):
    rng = np.random.default_rng(77)
    lens = rng.integers(100, 2000, size=12).astype(np.int32)
    lens[3] = 0                                    # a row that starts empty
    need = int(sum(-(-(int(n) + steps) // 16) for n in lens))
    max_pages = max(-(-(int(n) + steps) // 16) for n in lens)
    return wl.make_problem("ragged_cont", lens, Hq=16, Hkv=4, D=128, page_size=16,
                           num_pages=int(need * 1.25), max_pages=max_pages, rng=rng)


@pytest.mark.parametrize("case", ["continuous_one_split", "ragged_four_splits"])
def test_device_planned_steps_match_host_rules_and_oracle(case):
    steps = 60
    if case == "continuous_one_split":
        p = wl.continuous(steps=steps)
        splits = 1
    else:
        p = _ragged_problem(steps)
        splits = 4
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=splits)
    chunk = p.max_pages if splits == 1 else sess.plan.info()["chunk_pages"]
    sess.session.device_plan()
    rng = np.random.default_rng(5)
    k_h, v_h = p.k_pages, p.v_pages
    lens_h, table_h, free = p.seq_lens.copy(), p.block_table.copy(), list(p.free_pages)
    for step in range(steps):
        kn, vn = wl.new_tokens(rng, p.B, p.Hkv, p.D)
        sess.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
        _expected_reserve(lens_h, table_h, free, p.page_size)
        oracle.append(kn, vn, k_h, v_h, table_h, lens_h, inplace=True)
        if step in (0, 17, steps - 1):
            queue, order = sess.session.device_queue()
            want = oracle.enumerate_queue(lens_h, p.page_size, p.Hkv, chunk)
            assert np.array_equal(queue, want), step
            assert np.array_equal(order, _expected_order(want)), step
            assert np.array_equal(sess.table_h, table_h), step
            assert np.array_equal(sess.lens_h, lens_h), step
            ref = oracle.decode(p.q, k_h, v_h, table_h, lens_h, nthreads=16)
            assert_close(sess.out.cpu().numpy(), sess.lse.cpu().numpy(), *ref, what=f"{case} step {step}")
            assert sess.plan.status() == 0
    assert np.array_equal(sess.k.cpu().numpy().view(np.uint16), k_h)
    assert np.array_equal(sess.v.cpu().numpy().view(np.uint16), v_h)


def test_graph_captured_step_replays_like_eager_steps():
    steps = 40
    p = wl.continuous(steps=steps)
    rng = np.random.default_rng(6)
    toks = [wl.new_tokens(rng, p.B, p.Hkv, p.D) for _ in range(steps)]

    eager = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    eager.session.device_plan()
    for kn, vn in toks:
        eager.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
    torch.cuda.synchronize()
    e_out, e_lse = eager.out.cpu().numpy(), eager.lse.cpu().numpy()
    e_table, e_lens = eager.table_h, eager.lens_h
    del eager
    torch.cuda.empty_cache()

    graphed = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    graphed.session.device_plan()
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    # the first step runs eagerly (one-time kernel attribute set-up), the rest replay a graph
    kbuf.copy_(torch.from_numpy(toks[0][0].view(np.int16)))
    vbuf.copy_(torch.from_numpy(toks[0][1].view(np.int16)))
    graphed.step(kbuf, vbuf)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            graphed.step(kbuf, vbuf)
    torch.cuda.current_stream().wait_stream(side)
    for kn, vn in toks[1:]:
        kbuf.copy_(torch.from_numpy(kn.view(np.int16)))
        vbuf.copy_(torch.from_numpy(vn.view(np.int16)))
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(graphed.table_h, e_table)
    assert np.array_equal(graphed.lens_h, e_lens)
    assert np.array_equal(graphed.out.cpu().numpy(), e_out)
    assert np.array_equal(graphed.lse.cpu().numpy(), e_lse)
    assert graphed.plan.status() == 0
