"""Resident steps (pkv_resident_*) on the GPU: one cooperative kernel stays on
the device and runs each continuous-decoding step the host publishes.

Checked against the fp64 oracle at three steps (2e-3 / 1e-4), with the block
table, lengths and the whole K/V pool bit-exact against the oracle's append
after the run, and bit-identical to the same steps run as separate launches
(device-planned pkv_session_step): the resident kernel runs the same tile
code, and the last-arriver merge sums in split order.  The idle limit is made
to run out on purpose (a step that is never published) and must leave the
kernel with PKV_DEV_TIMEOUT and the context usable.
"""
import time

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


def _ragged_problem(steps):
    rng = np.random.default_rng(77)
    lens = rng.integers(100, 2000, size=12).astype(np.int32)
    lens[3] = 0                                    # a row that starts empty
    need = int(sum(-(-(int(n) + steps) // 16) for n in lens))
    max_pages = max(-(-(int(n) + steps) // 16) for n in lens)
    return wl.make_problem("ragged_cont", lens, Hq=16, Hkv=4, D=128, page_size=16,
                           num_pages=int(need * 1.25), max_pages=max_pages, rng=rng)


def _case(case, steps):
    if case == "continuous_one_split":
        return wl.continuous(steps=steps), 1
    return _ragged_problem(steps), 4


@pytest.mark.parametrize("case,math", [("continuous_one_split", "mma"), ("ragged_four_splits", "mma"),
                                       ("ragged_four_splits", "fma")])
def test_resident_steps_match_oracle_and_launched_steps(case, math):
    steps = 40
    check = (0, 17, steps - 1)
    p, splits = _case(case, steps)
    rng = np.random.default_rng(5)
    toks = [wl.new_tokens(rng, p.B, p.Hkv, p.D) for _ in range(steps)]

    # the same steps as separate launches
    eager = ContinuousSessions(p, force_mode="persistent", num_splits=splits, math=math)
    eager.session.device_plan()
    eager_out = {}
    for step, (kn, vn) in enumerate(toks):
        eager.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
        if step in check:
            eager_out[step] = (eager.out.cpu().numpy(), eager.lse.cpu().numpy())
    del eager
    torch.cuda.empty_cache()

    sess = ContinuousSessions(p, force_mode="persistent", num_splits=splits, math=math)
    sess.session.device_plan()
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    torch.cuda.synchronize()
    res = pkv.Resident(sess.session, sess.k, sess.v, sess.q, kbuf, vbuf, sess.out, sess.lse,
                       idle_limit_ns=5_000_000_000, times_cap=steps)
    got = {}
    try:
        for step, (kn, vn) in enumerate(toks):
            out_h = np.empty((p.B, p.Hq, p.D), np.float32) if step in check else None
            lse_h = np.empty((p.B, p.Hq), np.float32) if step in check else None
            res.step(k_new_h=kn.view(np.int16), v_new_h=vn.view(np.int16), out_h=out_h, lse_h=lse_h)
            if step in check:
                got[step] = (out_h, lse_h)
        with pytest.raises(pkv.PkvError):   # the session is busy while the kernel is resident
            sess.session.lengths()
    finally:
        res.stop()
    times = res.times()
    res.close()
    assert times.shape == (steps, 4) and np.all(np.diff(times.astype(np.int64), axis=1) >= 0)
    assert np.all(times[:, 3] > times[:, 0])
    assert sess.plan.status() == 0

    # the oracle replays the same steps on host copies
    k_h, v_h = p.k_pages.copy(), p.v_pages.copy()
    lens_h, table_h, free = p.seq_lens.copy(), p.block_table.copy(), list(p.free_pages)
    for step, (kn, vn) in enumerate(toks):
        _expected_reserve(lens_h, table_h, free, p.page_size)
        oracle.append(kn, vn, k_h, v_h, table_h, lens_h, inplace=True)
        if step in check:
            ref = oracle.decode(p.q, k_h, v_h, table_h, lens_h, nthreads=16)
            assert_close(*got[step], *ref, what=f"resident {case} step {step}")
            assert np.array_equal(got[step][0], eager_out[step][0]), step
            assert np.array_equal(got[step][1], eager_out[step][1]), step
    assert np.array_equal(sess.table_h, table_h)
    assert np.array_equal(sess.lens_h, lens_h)
    assert np.array_equal(sess.k.cpu().numpy().view(np.uint16), k_h)
    assert np.array_equal(sess.v.cpu().numpy().view(np.uint16), v_h)


def test_resident_idle_limit_runs_out_and_reports():
    p = wl.continuous(steps=4)
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    sess.session.device_plan()
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    torch.cuda.synchronize()
    res = pkv.Resident(sess.session, sess.k, sess.v, sess.q, kbuf, vbuf, sess.out, sess.lse,
                       idle_limit_ns=50_000_000)   # 50 ms
    time.sleep(0.5)                                # no step is published: the wait runs out
    with pytest.raises(pkv.PkvError) as e:
        res.stop()
    assert e.value.code == pkv.EDEVICE
    res.close()
    assert sess.plan.status() & pkv.DEV_TIMEOUT
    # the context and the session are still usable: one launched step against the oracle
    rng = np.random.default_rng(9)
    kn, vn = wl.new_tokens(rng, p.B, p.Hkv, p.D)
    sess.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
    k_h, v_h = p.k_pages.copy(), p.v_pages.copy()
    lens_h, table_h, free = p.seq_lens.copy(), p.block_table.copy(), list(p.free_pages)
    _expected_reserve(lens_h, table_h, free, p.page_size)
    oracle.append(kn, vn, k_h, v_h, table_h, lens_h, inplace=True)
    ref = oracle.decode(p.q, k_h, v_h, table_h, lens_h, nthreads=16)
    assert_close(sess.out.cpu().numpy(), sess.lse.cpu().numpy(), *ref, what="launched step after the timeout")
    assert sess.plan.status() == 0


def test_resident_yields_every_few_steps_and_lets_other_work_run():
    """yield_every = 7 over 40 steps: the kernel leaves the GPU after each 7th step
    of a launch and the next step launches it again (6 launches); its outputs are
    the launched steps' bit for bit, and while it is away another decode runs on
    the GPU and matches the oracle ("GPUOS", arXiv 2604.17861, set_yield_every)."""
    steps, every = 40, 7
    p = wl.continuous(steps=steps)
    rng = np.random.default_rng(12)
    toks = [wl.new_tokens(rng, p.B, p.Hkv, p.D) for _ in range(steps)]
    eager = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    eager.session.device_plan()
    for kn, vn in toks:
        eager.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
    torch.cuda.synchronize()
    e_out, e_lse = eager.out.cpu().numpy(), eager.lse.cpu().numpy()
    del eager
    torch.cuda.empty_cache()

    other = wl.tiny()
    other_ref = oracle.decode(other.q, other.k_pages, other.v_pages, other.block_table, other.seq_lens)
    other_dev = dict(q=torch.from_numpy(other.q.view(np.int16)).cuda(),
                     k=torch.from_numpy(other.k_pages.view(np.int16)).cuda(),
                     v=torch.from_numpy(other.v_pages.view(np.int16)).cuda(),
                     table=torch.from_numpy(other.block_table).cuda(), lens=torch.from_numpy(other.seq_lens).cuda(),
                     out=torch.empty((other.B, other.Hq, other.D), dtype=torch.float32, device="cuda"),
                     lse=torch.empty((other.B, other.Hq), dtype=torch.float32, device="cuda"))
    other_plan = pkv.Plan(other.seq_lens, other.block_table, other.page_size, B=other.B, Hq=other.Hq, Hkv=other.Hkv,
                          D=other.D, max_pages=other.max_pages, num_pages=other.num_pages, force_mode="split_queue",
                          num_splits=4)

    sess = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    sess.session.device_plan()
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    torch.cuda.synchronize()
    res = pkv.Resident(sess.session, sess.k, sess.v, sess.q, kbuf, vbuf, sess.out, sess.lse,
                       idle_limit_ns=5_000_000_000, times_cap=steps, yield_every=every)
    out_h = np.empty((p.B, p.Hq, p.D), np.float32)
    lse_h = np.empty((p.B, p.Hq), np.float32)
    try:
        for step, (kn, vn) in enumerate(toks):
            res.step(k_new_h=kn.view(np.int16), v_new_h=vn.view(np.int16), out_h=out_h, lse_h=lse_h)
            if step + 1 == 2 * every:   # the kernel has just yielded: the GPU runs other work
                pkv.decode(other_dev["q"], other_dev["k"], other_dev["v"], other_dev["table"], other_dev["lens"],
                           other_plan, other_dev["out"], other_dev["lse"])
                torch.cuda.synchronize()
                assert_close(other_dev["out"].cpu().numpy(), other_dev["lse"].cpu().numpy(), *other_ref,
                             what="decode between two resident launches")
        assert res.launches() == -(-steps // every)
    finally:
        res.stop()
    res.close()
    assert sess.plan.status() == 0
    assert np.array_equal(out_h, e_out) and np.array_equal(lse_h, e_lse)
