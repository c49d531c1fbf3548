"""Continuous sessions on the GPU: 56 sessions, 200 back-to-back steps of
append (one K/V token per session, a fresh page from the pool when one fills),
re-plan and persistent-queue decode.

Checked against the oracle at steps 0, 99 and 199 (2e-3 / 1e-4), with the
block table, lengths and the whole K/V pool bit-exact against the oracle's
append at the end.  The expected page assignment is rebuilt here from the
pool's rule (FIFO free list; a row takes a page when its next token starts
one), independently of the library.
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

CHECK_STEPS = (0, 99, 199)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _expected_reserve(lens, table, free, ps):
    for b in range(len(lens)):
        if lens[b] % ps == 0 and table[b, lens[b] // ps] < 0:
            table[b, lens[b] // ps] = free.pop(0)


@pytest.mark.parametrize("math", ["mma", "fma"])
def test_continuous_sessions(math):
    p = wl.continuous()
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=1, math=math)
    assert sess.plan.info()["mode_name"] == "persistent"
    rng = np.random.default_rng(wl.HELD_OUT_SEED + 1)
    k_h, v_h = p.k_pages, p.v_pages                 # host mirror, updated in place by the oracle
    lens_h = p.seq_lens.copy()
    table_h = p.block_table.copy()
    free = list(p.free_pages)
    for step in range(200):
        kn, vn = wl.new_tokens(rng, p.B, p.Hkv, p.D)
        sess.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
        _expected_reserve(lens_h, table_h, free, p.page_size)
        oracle.append(kn, vn, k_h, v_h, table_h, lens_h, inplace=True)
        if step in CHECK_STEPS:
            torch.cuda.synchronize()
            assert np.array_equal(sess.table_h, table_h), step
            assert np.array_equal(sess.lens_h, lens_h), step
            assert np.array_equal(sess.lens_d.cpu().numpy(), lens_h), step
            assert np.array_equal(sess.table_d.cpu().numpy(), table_h), step
            ref_out, ref_lse = oracle.decode(p.q, k_h, v_h, table_h, lens_h, nthreads=16)
            assert_close(sess.out.cpu().numpy(), sess.lse.cpu().numpy(), ref_out, ref_lse,
                         what=f"continuous step {step} {math}")
            assert sess.plan.status() == 0
    assert np.array_equal(sess.k.cpu().numpy().view(np.uint16), k_h)
    assert np.array_equal(sess.v.cpu().numpy().view(np.uint16), v_h)
    assert sess.pool.free_count() == len(free)


@pytest.mark.parametrize("route,splits", [("split_queue", 3), ("split_padded", 2), ("direct", 0)])
def test_session_steps_other_routes(route, splits):
    """Host-planned session steps on the non-persistent routes: the step's plan reaches
    the device through the append launch, and the queue route then reads it only after
    its grid dependency wait.  12 rows crossing page boundaries over 40 steps."""
    lens = np.array([15, 16, 17, 31, 32, 33, 1, 100, 250, 47, 64, 5], np.int32)
    steps = 40
    need = int(sum(-(-(int(n) + steps) // 16) for n in lens))
    max_pages = max(-(-(int(n) + steps) // 16) for n in lens)
    p = wl.make_problem("sess_routes", lens, Hq=16, Hkv=4, D=128, page_size=16, num_pages=need + 9,
                        max_pages=max_pages, seed=41)
    opts = dict(force_mode=route) if route == "direct" else dict(force_mode=route, num_splits=splits)
    sess = ContinuousSessions(p, **opts)
    rng = np.random.default_rng(42)
    k_h, v_h = p.k_pages, p.v_pages
    lens_h, table_h, free = p.seq_lens.copy(), p.block_table.copy(), list(p.free_pages)
    for step in range(steps):
        kn, vn = wl.new_tokens(rng, p.B, p.Hkv, p.D)
        sess.step(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda())
        _expected_reserve(lens_h, table_h, free, p.page_size)
        oracle.append(kn, vn, k_h, v_h, table_h, lens_h, inplace=True)
        if step in (0, 16, 39):
            torch.cuda.synchronize()
            assert np.array_equal(sess.table_d.cpu().numpy(), table_h), step
            assert np.array_equal(sess.lens_d.cpu().numpy(), lens_h), step
            assert_close(sess.out.cpu().numpy(), sess.lse.cpu().numpy(),
                         *oracle.decode(p.q, k_h, v_h, table_h, lens_h, nthreads=8),
                         what=f"{route} session step {step}")
            assert sess.plan.status() == 0
    assert np.array_equal(sess.k.cpu().numpy().view(np.uint16), k_h)
