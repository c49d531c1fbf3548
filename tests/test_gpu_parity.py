"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: max-abs 2e-3 on out, 1e-4 on LSE; work queues bit-exact against the
oracle's enumeration; device status word clean.  Covers every route, split
counts, ragged and edge lengths, every supported (D, G), and the full-size
workloads.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import (assert_close, expected_queue, make_plan, oracle_result, run, to_device)

pytestmark = pytest.mark.gpu

ROUTES = ["direct", "split_queue", "split_padded", "persistent"]
MATHS = ["fma", "mma"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


COPIES = ["lsu", "tma"]


@pytest.mark.parametrize("copy", COPIES)
@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("splits", [1, 2, 4])
def test_tiny_every_route_and_split(route, splits, math, copy):
    p = wl.tiny()
    ref = oracle_result(p)
    out, lse, plan, _ = run(p, force_mode=route, num_splits=splits, math=math, copy=copy)
    assert_close(out, lse, *ref, what=f"tiny {route} S={splits} {math} {copy}")
    info = plan.info()
    assert info["mode_name"] == route
    assert np.array_equal(plan.queue(), expected_queue(p, info))
    assert plan.status() == 0


@pytest.mark.parametrize("math", MATHS)
def test_tiny_split_partials_match_oracle_partials(math):
    """The partial kernel's per-tile states equal the oracle's split partials."""
    p = wl.tiny()
    _, _, plan, _ = run(p, force_mode="split_queue", num_splits=4, math=math)
    o, lse = plan.read_workspace()
    q = plan.queue()
    for slot, (b, kvh, s, pb, pe) in enumerate(q):
        ro, rl = oracle.partial(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, b, kvh,
                                pb * p.page_size, pe * p.page_size)
        assert np.max(np.abs(o[slot] - ro)) <= 2e-3
        assert np.max(np.abs(lse[slot] - rl)) <= 1e-4


EDGE_LENS = [1, 15, 16, 17, 32, 33, 0, 250]


@pytest.mark.parametrize("copy", COPIES)
@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("splits", [1, 3, 16])
def test_edge_lengths(route, splits, math, copy):
    p = wl.make_problem("edges", EDGE_LENS, Hq=8, Hkv=2, D=128, page_size=16, num_pages=48, seed=21)
    ref = oracle_result(p)
    out, lse, plan, _ = run(p, force_mode=route, num_splits=splits, math=math, copy=copy)
    assert_close(out, lse, *ref, what=f"edges {route} S={splits} {math} {copy}")
    assert np.array_equal(plan.queue(), expected_queue(p, plan.info()))
    assert plan.status() == 0


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_every_head_shape(D, G, math):
    Hkv = 2
    p = wl.make_problem(f"shape{D}x{G}", [77, 300, 16], Hq=G * Hkv, Hkv=Hkv, D=D, page_size=16,
                        num_pages=40, seed=22)
    ref = oracle_result(p)
    for route, splits in [("direct", 0), ("split_queue", 5), ("persistent", 3)]:
        out, lse, _, _ = run(p, force_mode=route, num_splits=splits, math=math)
        assert_close(out, lse, *ref, what=f"D={D} G={G} {route} {math}")


@pytest.mark.parametrize("route", ["split_queue", "split_padded", "persistent"])
def test_separate_merge_launch(route):
    """The merge as its own kernel gives the same result as the fused last-arriver merge."""
    p = wl.make_problem("sepmerge", EDGE_LENS, Hq=8, Hkv=2, D=128, page_size=16, num_pages=48, seed=26)
    ref = oracle_result(p)
    out, lse, plan, _ = run(p, force_mode=route, num_splits=4, separate_merge=True)
    assert plan.info()["launches_per_step"] == 2
    assert_close(out, lse, *ref, what=f"separate merge {route}")
    out2, lse2, plan2, _ = run(p, force_mode=route, num_splits=4)
    assert plan2.info()["launches_per_step"] == 1
    assert_close(out2, lse2, *ref, what=f"fused merge {route}")
    # the two merges sum in different orders; they agree far inside the tolerance
    assert np.max(np.abs(out - out2)) <= 1e-5
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lse2)) and np.max(np.abs(lse[fin] - lse2[fin])) <= 1e-5


@pytest.mark.parametrize("copy", COPIES)
@pytest.mark.parametrize("page_size", [32, 64, 128, 256])
def test_larger_pages(page_size, copy):
    p = wl.make_problem("pages", [1, 63, 64, 65, 500], Hq=8, Hkv=2, D=128, page_size=page_size,
                        num_pages=24, seed=23)
    ref = oracle_result(p)
    for route in ROUTES:
        out, lse, _, _ = run(p, force_mode=route, num_splits=3, copy=copy)
        assert_close(out, lse, *ref, what=f"ps={page_size} {route} {copy}")


MERGES = ["last", "all"]


@pytest.mark.parametrize("merge", MERGES)
@pytest.mark.parametrize("route", ["split_queue", "split_padded"])
@pytest.mark.parametrize("splits", [2, 3, 16])
def test_fused_merge_kinds(route, splits, merge):
    """Both fused merges (last arriver; every split sharing out the outputs) match
    the oracle, and their counters rewind: repeated launches give the same bits."""
    p = wl.make_problem("merges", EDGE_LENS, Hq=8, Hkv=2, D=128, page_size=16, num_pages=48, seed=27)
    ref = oracle_result(p)
    out, lse, plan, dev = run(p, force_mode=route, num_splits=splits, merge=merge)
    assert plan.info()["merge_name"] == merge
    assert_close(out, lse, *ref, what=f"{merge} merge {route} S={splits}")
    for _ in range(2):
        out2, lse2, _, _ = run(p, dev=dev, plan=plan)
        assert np.array_equal(out2, out) and np.array_equal(lse2, lse)
    assert plan.status() == 0


@pytest.mark.parametrize("merge", MERGES)
@pytest.mark.parametrize("Hq,D", [(8, 128), (16, 128), (2, 64)])
def test_fused_merge_more_splits_than_lanes(merge, Hq, D):
    """64 splits of one (row, KV head): more than a warp's lanes; with G = 1 and
    D = 64 also more splits than float4 outputs, so some splits merge nothing."""
    p = wl.make_problem("manysplits", [4096, 1000, 17, 0], Hq=Hq, Hkv=2, D=D, page_size=16,
                        num_pages=360, seed=28)
    ref = oracle_result(p)
    out, lse, plan, _ = run(p, force_mode="split_queue", num_splits=64, merge=merge)
    info = plan.info()
    assert info["merge_name"] == merge and info["max_splits"] == 64
    assert_close(out, lse, *ref, what=f"{merge} merge, 64 splits")
    assert plan.status() == 0


@pytest.mark.parametrize("Hq,D,splits", [(16, 128, 16), (2, 64, 16), (4, 64, 40), (16, 64, 24), (2, 128, 16),
                                          (8, 128, 40)])
def test_last_merge_group_sizes(Hq, D, splits):
    """The last arriver's chunked merge for every lanes-per-output split (G*D/4
    outputs over 256 threads: 1, 2, 8 or 16 lanes each) and up to 7 chunks;
    repeated launches give the same bits."""
    p = wl.make_problem("groups", [4096, 1000, 17, 0], Hq=Hq, Hkv=2, D=D, page_size=16, num_pages=360, seed=30)
    ref = oracle_result(p)
    out, lse, plan, dev = run(p, force_mode="split_queue", num_splits=splits, merge="last")
    assert_close(out, lse, *ref, what=f"Hq={Hq} D={D} S={splits}")
    out2, lse2, _, _ = run(p, dev=dev, plan=plan)
    assert np.array_equal(out2, out) and np.array_equal(lse2, lse)
    assert plan.status() == 0


@pytest.mark.parametrize("Hq,D", [(8, 128), (16, 128), (2, 64)])
def test_fused_merge_beyond_64_splits(Hq, D):
    """86 splits of the 4096-token row (3 pages each): past the register merge's
    64, so the last arriver stages the partials in shared memory (the ALL merge
    refuses more than 64 splits)."""
    merge = "last"
    p = wl.make_problem("splits86", [4096, 1000, 17, 0], Hq=Hq, Hkv=2, D=D, page_size=16,
                        num_pages=360, seed=29)
    ref = oracle_result(p)
    out, lse, plan, dev = run(p, force_mode="split_queue", num_splits=96, merge=merge)
    info = plan.info()
    assert info["merge_name"] == merge and info["max_splits"] == 86, info["max_splits"]
    assert_close(out, lse, *ref, what=f"{merge} merge, 86 splits")
    out2, lse2, _, _ = run(p, dev=dev, plan=plan)
    assert np.array_equal(out2, out) and np.array_equal(lse2, lse)
    assert plan.status() == 0


@pytest.mark.parametrize("merge", MERGES)
def test_bad_page_poisons_through_either_merge(merge):
    p = wl.tiny()
    bad = p.block_table.copy()
    bad[1, 2] = p.num_pages + 5
    p_bad = wl.Problem("bad", p.q, p.k_pages, p.v_pages, bad, p.seq_lens, p.page_size)
    for route in ["split_queue", "split_padded"]:
        out, lse, plan, _ = run(p_bad, host_table=False, force_mode=route, num_splits=4, merge=merge)
        assert plan.status() & pkv.DEV_PAGE_OOB, route
        assert np.all(np.isnan(out[1])) and np.all(np.isnan(lse[1])), route
        assert np.all(np.isfinite(out[0])), route


def test_all_rows_empty():
    p = wl.make_problem("empty", [0, 0, 0], Hq=4, Hkv=1, D=64, page_size=16, num_pages=4, seed=24)
    for route in ROUTES:
        out, lse, _, _ = run(p, force_mode=route, num_splits=2)
        assert np.array_equal(out, np.zeros_like(out)) and np.all(np.isneginf(lse)), route


def test_permuted_block_table_same_result():
    p = wl.mixed()
    out0, lse0, _, _ = run(p, force_mode="split_queue", num_splits=8)
    rng = np.random.default_rng(25)
    perm = rng.permutation(p.num_pages)
    k2 = np.empty_like(p.k_pages)
    v2 = np.empty_like(p.v_pages)
    k2[perm] = p.k_pages
    v2[perm] = p.v_pages
    t2 = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    p2 = wl.Problem("mixed_perm", p.q, k2, v2, t2, p.seq_lens, p.page_size)
    out1, lse1, _, _ = run(p2, force_mode="split_queue", num_splits=8)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_deterministic_across_runs():
    p = wl.mixed()
    for route in ["persistent", "split_padded"]:
        dev = to_device(p)
        plan = make_plan(p, force_mode=route)
        a = run(p, dev=dev, plan=plan)[:2]
        a = (a[0].copy(), a[1].copy())
        b = run(p, dev=dev, plan=plan)[:2]
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), route


def test_back_to_back_launches_of_different_plans():
    """Decodes of different plans queued back to back on one stream, with no host
    synchronisation between them: each launch may start while the previous one
    finishes (programmatic dependent launch), reads its own host-staged queue
    entry early, and everything else only after the dependency wait; the clones
    between the decodes read what the previous decode wrote."""
    pa = wl.make_problem("b2b_a", [700, 33, 1500], Hq=16, Hkv=4, D=128, page_size=16, num_pages=200, seed=31)
    pb = wl.mixed()
    da, db = to_device(pa), to_device(pb)
    plans = [make_plan(pa, force_mode="split_queue", num_splits=8), make_plan(pb),
             make_plan(pa, force_mode="persistent", num_splits=3)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pkv.decode(da["q"], da["k"], da["v"], da["table"], da["lens"], plans[0], da["out"], da["lse"], stream=stream)
        out0 = da["out"].clone()
        pkv.decode(db["q"], db["k"], db["v"], db["table"], db["lens"], plans[1], db["out"], db["lse"], stream=stream)
        out1, lse1 = db["out"].clone(), db["lse"].clone()
        pkv.decode(da["q"], da["k"], da["v"], da["table"], da["lens"], plans[2], da["out"], da["lse"], stream=stream)
    stream.synchronize()
    ref_a, ref_b = oracle_result(pa), oracle_result(pb)
    assert np.max(np.abs(out0.cpu().numpy() - ref_a[0])) <= 2e-3
    assert_close(out1.cpu().numpy(), lse1.cpu().numpy(), *ref_b, what="second of three")
    assert_close(da["out"].cpu().numpy(), da["lse"].cpu().numpy(), *ref_a, what="third of three")
    for plan in plans:
        assert plan.status() == 0


def _host_buffers(p, kind):
    """q / out / lse host buffers: pinned (the kernel uses them in place), pageable
    numpy arrays (staged through the plan's pinned buffer), or pinned tensors whose
    address is 4 bytes past a 16-byte boundary (staged too: the kernel's vector
    accesses need 16-byte alignment)."""
    q = p.q.view(np.int16)
    if kind == "pageable":
        return q.copy(), np.empty((p.B, p.Hq, p.D), np.float32), np.empty((p.B, p.Hq), np.float32)
    if kind == "pinned":
        return (torch.from_numpy(q).pin_memory(), torch.empty((p.B, p.Hq, p.D), dtype=torch.float32).pin_memory(),
                torch.empty((p.B, p.Hq), dtype=torch.float32).pin_memory())
    qb = torch.empty(q.size + 2, dtype=torch.int16).pin_memory()
    q_h = qb[2:].view(p.B, p.Hq, p.D)
    q_h.copy_(torch.from_numpy(q))
    out_h = torch.empty(p.B * p.Hq * p.D + 1, dtype=torch.float32).pin_memory()[1:].view(p.B, p.Hq, p.D)
    lse_h = torch.empty(p.B * p.Hq + 1, dtype=torch.float32).pin_memory()[1:].view(p.B, p.Hq)
    assert q_h.data_ptr() % 16 == 4 and out_h.data_ptr() % 16 == 4
    return q_h, out_h, lse_h


def _np(a):
    return a.numpy() if isinstance(a, torch.Tensor) else a


@pytest.mark.parametrize("kind", ["pinned", "pageable", "misaligned"])
@pytest.mark.parametrize("route", ["split_queue", "direct", "persistent"])
def test_decode_with_host_buffers(route, kind):
    """pkv_decode_host: q from host memory, out / lse back to host memory."""
    p = wl.make_problem("host_bufs", [700, 33, 1500, 0], Hq=16, Hkv=4, D=128, page_size=16, num_pages=200, seed=33)
    dev = to_device(p)
    plan = make_plan(p, force_mode=route, num_splits=5)
    q_h, out_h, lse_h = _host_buffers(p, kind)
    pkv.decode_host(q_h, dev["k"], dev["v"], dev["table"], dev["lens"], plan, out_h, lse_h)
    assert_close(_np(out_h), _np(lse_h), *oracle_result(p), what=f"host buffers {route} {kind}")
    out, lse, _, _ = run(p, dev=dev, plan=plan)
    assert np.array_equal(out, _np(out_h)) and np.array_equal(lse, _np(lse_h))
    assert plan.status() == 0


@pytest.mark.parametrize("route", ["split_queue", "persistent"])
def test_host_buffers_after_replanning(route):
    """A re-planned queue is read in place from the plan's pinned host copy by
    pkv_decode_host and uploaded by the next pkv_decode; both agree with the oracle
    for the new lengths, and a second host-buffer decode (plan now uploaded) too."""
    p = wl.make_problem("replan", [700, 33, 1500, 0], Hq=16, Hkv=4, D=128, page_size=16, num_pages=200, seed=34)
    dev = to_device(p)
    plan = make_plan(p, force_mode=route, num_splits=5)
    q_h, out_h, lse_h = _host_buffers(p, "pinned")
    pkv.decode_host(q_h, dev["k"], dev["v"], dev["table"], dev["lens"], plan, out_h, lse_h)
    assert_close(out_h.numpy(), lse_h.numpy(), *oracle_result(p), what="before re-plan")
    lens2 = np.array([650, 40, 1401, 0], np.int32)
    p2 = wl.Problem("replan2", p.q, p.k_pages, p.v_pages, p.block_table, lens2, p.page_size)
    ref2 = oracle_result(p2)
    dev["lens"].copy_(torch.from_numpy(lens2))
    plan.update(lens2, p.block_table)
    pkv.decode_host(q_h, dev["k"], dev["v"], dev["table"], dev["lens"], plan, out_h, lse_h)   # plan read in place
    assert_close(out_h.numpy(), lse_h.numpy(), *ref2, what="host buffers after re-plan")
    first = (out_h.numpy().copy(), lse_h.numpy().copy())
    out, lse, _, _ = run(p2, dev=dev, plan=plan)   # uploads the new plan
    assert np.array_equal(out, first[0]) and np.array_equal(lse, first[1])
    out_h.fill_(float("nan"))
    pkv.decode_host(q_h, dev["k"], dev["v"], dev["table"], dev["lens"], plan, out_h, lse_h)   # uploaded plan
    assert np.array_equal(out_h.numpy(), first[0]) and np.array_equal(lse_h.numpy(), first[1])
    assert plan.status() == 0


def test_bad_page_id_flags_status_and_poisons():
    """A table entry outside the pool (the planner is not shown the table) is caught in
    the kernel: status bit set, output NaN, no access through the bad id."""
    p = wl.tiny()
    bad = p.block_table.copy()
    bad[1, 2] = p.num_pages + 5
    p_bad = wl.Problem("bad", p.q, p.k_pages, p.v_pages, bad, p.seq_lens, p.page_size)
    for route, copy in [(r, c) for r in ROUTES for c in COPIES]:
        out, lse, plan, _ = run(p_bad, host_table=False, force_mode=route, num_splits=2, copy=copy)
        assert plan.status() & pkv.DEV_PAGE_OOB, route
        assert np.all(np.isnan(out[1])), route
        assert np.all(np.isfinite(out[0])), route


def test_plan_mismatch_is_detected():
    p = wl.tiny()
    plan = make_plan(p, force_mode="split_queue", num_splits=2)
    dev = to_device(p)
    dev["lens"] = torch.tensor([37, 60], dtype=torch.int32, device="cuda")   # not what was planned
    pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
    assert plan.status() & pkv.DEV_PLAN_MISMATCH


def test_host_validation_errors():
    p = wl.tiny()
    bad = p.block_table.copy()
    bad[0, 1] = -3
    with pytest.raises(pkv.PkvError) as e:
        make_plan(wl.Problem("b", p.q, p.k_pages, p.v_pages, bad, p.seq_lens, p.page_size))
    assert e.value.code == pkv.EINVAL


# --- the full-size workloads ---------------------------------------------------------

@pytest.fixture(scope="module")
def batch1_long_ref():
    p = wl.batch1_long()
    return p, oracle_result(p, nthreads=16)


@pytest.fixture(scope="module")
def mixed_ref():
    p = wl.mixed()
    return p, oracle_result(p, nthreads=16)


@pytest.mark.parametrize("math,copy,merge", [("fma", "lsu", "auto"), ("mma", "lsu", "auto"), ("mma", "tma", "auto"),
                                             ("mma", "lsu", "last")])
@pytest.mark.parametrize("route", ["split_queue", "persistent"])
def test_batch1_long_32k(route, math, copy, merge, batch1_long_ref):
    p, ref = batch1_long_ref
    out, lse, plan, _ = run(p, force_mode=route, num_splits=32, math=math, copy=copy, merge=merge)
    assert_close(out, lse, *ref, what=f"batch1_long {route} {math} {copy} {merge}")
    info = plan.info()
    assert info["chunk_pages"] == 64 and info["num_work_items"] == 256
    assert np.array_equal(plan.queue(), expected_queue(p, info))
    assert plan.status() == 0


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("route", ["split_queue", "split_padded", "persistent", "auto"])
def test_mixed_batch(route, math, mixed_ref):
    p, ref = mixed_ref
    out, lse, plan, _ = run(p, force_mode=route, math=math)
    assert_close(out, lse, *ref, what=f"mixed {route} {math}")
    assert np.array_equal(plan.queue(), expected_queue(p, plan.info()))
    assert plan.status() == 0


def test_high_batch_policy_chooses_direct():
    p = wl.high_batch()
    ref = oracle_result(p, nthreads=16)
    dev = to_device(p)
    for math in MATHS:
        out, lse, plan, _ = run(p, dev=dev, math=math)
        assert plan.info()["mode_name"] == "direct"
        assert plan.info()["launches_per_step"] == 1
        assert_close(out, lse, *ref, what=f"high_batch {math}")
        assert plan.status() == 0
