"""Slot admit / evict at step boundaries (pkv_session_evict / pkv_session_admit,
pkv_resident_evict / pkv_resident_admit) on the GPU.

60 continuous steps of 12 sessions; at steps 10, 12, 30 and 45 sessions leave
(their pages go back to the free list) and new ones arrive in the freed slots
with a prompt written into fresh pages ("WPK persistent kernel", dotwave.ai,
"What has to exist instead": fixed arenas, slots reset at a beat boundary).
Every mode is run: host-planned steps, device-planned steps, a device-planned
step captured once in a CUDA graph and replayed across the changes (no
re-capture), and one resident kernel for all steps.  At four steps the decode
must match the fp64 oracle on the oracle slot model's pages (2e-3 / 1e-4; idle
slots decode to out 0, lse -inf); the block table, lengths, active flags and
the free list (front first) must equal the model's bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.slots import SlotModel
from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from paged_kv_decode_block_gb300.session import ContinuousSessions
from pkv_testutil import assert_close

pytestmark = pytest.mark.gpu

STEPS = 60
CHECK = (11, 31, 46, 59)
# boundary before step -> (evictions, (admitted rows, prompt lengths))
EVENTS = {10: ([3, 7], None), 12: ([], ([7], [50])), 30: ([0, 5, 11], ([3, 0], [100, 17])),
          45: ([], ([5, 11], [33, 64]))}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _problem():
    rng = np.random.default_rng(91)
    lens = rng.integers(40, 300, size=12).astype(np.int32)
    return wl.make_problem("slots", lens, Hq=8, Hkv=2, D=64, page_size=16, num_pages=420, max_pages=32, rng=rng)


def _inputs(p):
    rng = np.random.default_rng(92)
    toks = [wl.new_tokens(rng, p.B, p.Hkv, p.D) for _ in range(STEPS)]
    prompts = {}
    for step, (_, adm) in EVENTS.items():
        if adm:
            n = int(sum(adm[1]))
            prompts[step] = (wl.bf16_normal(rng, (n, p.Hkv, p.D)), wl.bf16_normal(rng, (n, p.Hkv, p.D)))
    return toks, prompts


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _model_check(p, model, out, lse, what):
    ref = oracle.decode(p.q, model.k_pages, model.v_pages, model.table, model.lens, nthreads=8)
    assert_close(out, lse, *ref, what=what)


def _state_check(sess, model, what):
    assert np.array_equal(sess.session.table(), model.table), what
    assert np.array_equal(sess.session.lengths(), model.lens), what
    free, active = sess.session.free_pages()
    assert np.array_equal(active, model.active), what
    assert free.tolist() == list(model.free), what


@pytest.mark.parametrize("mode", ["host", "device", "graph"])
def test_slots_across_launched_steps(mode):
    p = _problem()
    toks, prompts = _inputs(p)
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    model = SlotModel(p.seq_lens, p.block_table, p.free_pages, p.page_size, p.k_pages.copy(), p.v_pages.copy())
    if mode != "host":
        sess.session.device_plan()
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    graph = None
    keep = []
    for step in range(STEPS):
        if step in EVENTS:
            evict, adm = EVENTS[step]
            if evict:
                sess.session.evict(evict)
                model.evict(evict)
            if adm:
                kp, vp = prompts[step]
                kd, vd = _dev(kp), _dev(vp)
                keep.append((kd, vd))
                sess.session.admit(adm[0], adm[1], kd, vd, sess.k, sess.v)
                model.admit(adm[0], adm[1], kp, vp)
        kn, vn = toks[step]
        kbuf.copy_(_dev(kn))
        vbuf.copy_(_dev(vn))
        if graph is not None:
            graph.replay()
        else:
            sess.step(kbuf, vbuf)
        model.step(kn, vn)
        if mode == "graph" and graph is None:   # the first step ran eagerly; capture the step once
            torch.cuda.synchronize()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(graph, stream=side):
                    sess.step(kbuf, vbuf)
            torch.cuda.current_stream().wait_stream(side)
        if step in CHECK:
            torch.cuda.synchronize()
            _model_check(p, model, sess.out.cpu().numpy(), sess.lse.cpu().numpy(), f"{mode} step {step}")
            _state_check(sess, model, f"{mode} step {step}")
            idle = np.nonzero(model.active == 0)[0]
            assert np.all(sess.out.cpu().numpy()[idle] == 0) and np.all(np.isneginf(sess.lse.cpu().numpy()[idle]))
    torch.cuda.synchronize()
    assert np.array_equal(sess.k.cpu().numpy().view(np.uint16), model.k_pages)
    assert np.array_equal(sess.v.cpu().numpy().view(np.uint16), model.v_pages)
    assert sess.plan.status() == 0


def test_slots_through_a_resident_kernel():
    p = _problem()
    toks, prompts = _inputs(p)
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    sess.session.device_plan()
    model = SlotModel(p.seq_lens, p.block_table, p.free_pages, p.page_size, p.k_pages.copy(), p.v_pages.copy())
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    torch.cuda.synchronize()
    res = pkv.Resident(sess.session, sess.k, sess.v, sess.q, kbuf, vbuf, sess.out, sess.lse,
                       idle_limit_ns=5_000_000_000, times_cap=STEPS)
    got = {}
    try:
        for step in range(STEPS):
            if step in EVENTS:
                evict, adm = EVENTS[step]
                if evict:
                    res.evict(evict)
                    model.evict(evict)
                if adm:
                    kp, vp = prompts[step]
                    res.admit(adm[0], adm[1], _dev(kp), _dev(vp))
                    model.admit(adm[0], adm[1], kp, vp)
            kn, vn = toks[step]
            out_h = np.empty((p.B, p.Hq, p.D), np.float32) if step in CHECK else None
            lse_h = np.empty((p.B, p.Hq), np.float32) if step in CHECK else None
            res.step(k_new_h=kn.view(np.int16), v_new_h=vn.view(np.int16), out_h=out_h, lse_h=lse_h)
            model.step(kn, vn)
            if step in CHECK:
                got[step] = (out_h, lse_h, model.k_pages.copy(), model.v_pages.copy(), model.table.copy(),
                             model.lens.copy())
    finally:
        res.stop()
    res.close()
    assert sess.plan.status() == 0
    for step, (out_h, lse_h, k, v, table, lens) in got.items():
        ref = oracle.decode(p.q, k, v, table, lens, nthreads=8)
        assert_close(out_h, lse_h, *ref, what=f"resident step {step}")
    _state_check(sess, model, "resident, after the run")
    assert np.array_equal(sess.k.cpu().numpy().view(np.uint16), model.k_pages)
    assert np.array_equal(sess.v.cpu().numpy().view(np.uint16), model.v_pages)


def test_slot_calls_refuse_bad_requests_and_change_nothing():
    # three rows (3, 4 and 7 pages) and a pool with 5 pages to spare
    p = wl.make_problem("slots_small", [40, 60, 100], Hq=8, Hkv=2, D=64, page_size=16, num_pages=19,
                        max_pages=32, seed=93)
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=1)
    s = sess.session
    free0, active0 = s.free_pages()
    table0, lens0 = s.table(), s.lengths()
    assert len(free0) == 5 and active0.tolist() == [1, 1, 1]
    kd = torch.zeros((600, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    for call in (lambda: s.evict([3]), lambda: s.evict([1, 1]), lambda: s.evict([-1]),
                 lambda: s.admit([2], [10], kd, kd, sess.k, sess.v)):   # out of range, twice, active row
        with pytest.raises(pkv.PkvError) as e:
            call()
        assert e.value.code == pkv.EINVAL
    free, active = s.free_pages()
    assert free.tolist() == free0.tolist() and active.tolist() == [1, 1, 1]
    s.evict([0])                                   # 3 pages back: 8 free
    free1, active1 = s.free_pages()
    assert active1.tolist() == [0, 1, 1] and free1.tolist() == free0.tolist() + table0[0, :3].tolist()
    for lens, code in (([-1], pkv.EINVAL), ([32 * 16 + 1], pkv.EINVAL), ([9 * 16], pkv.ENOSPACE)):
        with pytest.raises(pkv.PkvError) as e:     # negative, longer than the table, more pages than free
            s.admit([0], lens, kd, kd, sess.k, sess.v)
        assert e.value.code == code
    with pytest.raises(pkv.PkvError) as e:         # a row evicted twice
        s.evict([0])
    assert e.value.code == pkv.EINVAL
    free2, active2 = s.free_pages()
    assert free2.tolist() == free1.tolist() and active2.tolist() == [0, 1, 1]
    assert np.array_equal(s.table()[1:], table0[1:]) and np.all(s.table()[0] == -1)
    assert s.lengths().tolist() == [0] + lens0[1:].tolist()
    s.admit([0], [8 * 16], kd, kd, sess.k, sess.v)  # exactly what is free
    assert len(s.free_pages()[0]) == 0 and s.lengths()[0] == 128
