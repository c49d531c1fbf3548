"""Host-side checks that need no GPU: the C ABI library loads and exports every
declared symbol, the planner's tile queue equals the oracle's enumeration bit
for bit, the policy's route choices, validation errors, and the page pool.

Planner reading: "PersistentKV" (gist.science summary), Methodology section 1
("Sequence Splitting", "Row-Local Bounds", "Compact Workqueue") and section 2
("Calibrated Adaptive Policy").
"""
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
NUM_SMS = 152


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_block_gb300.csrc import build
    build.build()
    return pkv.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = pkv.load()
    names = _declared_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding describes exactly the declared ABI
    assert set(pkv.SIGNATURES) == set(names)


def _dry(p, **opts):
    return pkv.dry_run(p.seq_lens, p.block_table, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                       max_pages=p.max_pages, num_pages=p.num_pages, num_sms=NUM_SMS, **opts)


def _geom_problem(lens, Hq=8, Hkv=2, D=64, ps=16, slack=4, seed=0):
    lens = np.asarray(lens, np.int32)
    max_pages = max(1, int(max(-(-int(n) // ps) for n in lens)) + slack)
    B = len(lens)
    table = np.full((B, max_pages), -1, np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        P = -(-int(n) // ps)
        table[b, :P] = np.arange(nxt, nxt + P)
        nxt += P
    return wl.Problem("geom", np.zeros((B, Hq, D), np.uint16), np.zeros((max(nxt, 1), ps, Hkv, D), np.uint16),
                      np.zeros((max(nxt, 1), ps, Hkv, D), np.uint16), table, lens, ps)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("mode", ["split_queue", "persistent", "split_padded"])
def test_planner_queue_bit_exact_against_oracle_enumeration(seed, mode):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 12))
    lens = rng.integers(0, 3000, size=B)
    if seed == 0:
        lens[:] = 0
    p = _geom_problem(lens, Hkv=int(rng.choice([1, 2, 8])), Hq=8, seed=seed)
    S = int(rng.integers(1, 40))
    info, items = _dry(p, force_mode=mode, num_splits=S)
    C = oracle.chunk_pages_for_splits(p.seq_lens, p.page_size, S)
    assert info["chunk_pages"] == C
    if mode == "split_padded":
        want = oracle.enumerate_padded_grid(p.seq_lens, p.page_size, p.Hkv, C)
        if want.size == 0:   # an all-empty batch still has one neutral slot per (row, KV head)
            want = oracle.enumerate_padded_grid(np.ones(B, np.int32) * 0, p.page_size, p.Hkv, 1)
            want = np.array([(b, h, 0, 0, 0) for b in range(B) for h in range(p.Hkv)], np.int32).reshape(-1, 5)
        assert info["empty_tiles"] == int(np.sum(want[:, 3] == want[:, 4]))
    else:
        want = oracle.enumerate_queue(p.seq_lens, p.page_size, p.Hkv, C)
    assert items.dtype == np.int32 and np.array_equal(items, want)
    assert info["num_work_items"] == len(want)


def test_workload_policies():
    tiny = wl.tiny()
    info, q = _dry(tiny)
    # 7 pages fit one chunk: one queue tile per row, finalised in place
    assert (info["mode_name"], info["chunk_pages"], info["max_splits"]) == ("split_queue", 8, 1)
    assert np.array_equal(q, oracle.enumerate_queue(tiny.seq_lens, 16, 1, 8))
    for S, C in [(1, 7), (2, 4), (4, 2)]:
        info, q = _dry(tiny, force_mode="split_queue", num_splits=S)
        assert info["chunk_pages"] == C
        assert np.array_equal(q, oracle.enumerate_queue(tiny.seq_lens, 16, 1, C))

    # batch-1 long context: 32 splits of 64 pages, 8 x 32 tiles, one launch (fused merge)
    b1 = _geom_problem([32768], Hq=32, Hkv=8, D=128)
    info, q = _dry(b1, num_splits=32)
    assert (info["mode_name"], info["chunk_pages"], info["num_work_items"]) == ("split_queue", 64, 256)
    assert info["launches_per_step"] == 1
    assert info["kv_bytes"] == 134217728
    info, _ = _dry(b1)   # the policy alone also splits a lone long row
    assert info["mode_name"] == "split_queue" and info["num_work_items"] >= NUM_SMS

    # mixed small batch: compact queue; the padded grid holds the same tiles plus empty slots
    lens, _ = wl.mixed_lengths()
    mixed = _geom_problem(lens, Hq=32, Hkv=8, D=128)
    qi, qq = _dry(mixed)
    assert qi["mode_name"] == "split_queue"
    pi, pq = _dry(mixed, force_mode="split_padded")
    assert pi["num_work_items"] == 8 * 8 * pi["max_splits"]
    assert pi["empty_tiles"] == pi["num_work_items"] - qi["num_work_items"]
    assert np.array_equal(pq[pq[:, 3] < pq[:, 4]], qq)

    # high batch: 64 x 8 units fill the SMs, so the policy must choose the direct kernel
    hb = _geom_problem([4096] * 64, Hq=32, Hkv=8, D=128)
    info, q = _dry(hb)
    assert info["mode_name"] == "direct" and info["launches_per_step"] == 1 and len(q) == 512

    # continuous sessions run the persistent queue, one split per session
    cont = _geom_problem(np.random.default_rng(1).integers(1024, 8193, 56), Hq=32, Hkv=8, D=128, slack=13)
    info, q = _dry(cont, force_mode="persistent", num_splits=1, ctas_per_sm=2)
    assert info["mode_name"] == "persistent" and len(q) == 56 * 8
    assert info["grid_ctas"] == min(len(q), 2 * NUM_SMS)


def test_copy_engine_resolution():
    """copy=auto takes TMA boxes on the one-tile-per-CTA routes and cp.async on the
    persistent route; an explicit choice is kept."""
    b1 = _geom_problem([32768], Hq=32, Hkv=8, D=128)
    for route, want in (("split_queue", "tma"), ("split_padded", "tma"), ("direct", "tma"), ("persistent", "lsu")):
        info, _ = _dry(b1, force_mode=route, num_splits=32, ctas_per_sm=2)
        assert (info["mode_name"], info["copy_name"]) == (route, want)
        for forced in ("lsu", "tma"):
            info, _ = _dry(b1, force_mode=route, num_splits=32, ctas_per_sm=2, copy=forced)
            assert info["copy_name"] == forced


def test_plan_info_layout_matches_the_header():
    """The binding's pkv_plan_info is the header's struct: its size is checked by a dry
    run writing a full struct, with a guard word past the end left alone."""
    import ctypes
    b1 = _geom_problem([4096], Hq=32, Hkv=8, D=128)
    lib = pkv.load()
    lens = np.ascontiguousarray(b1.seq_lens, np.int32)

    class Guarded(ctypes.Structure):
        _fields_ = [("info", pkv.PlanInfo), ("guard", ctypes.c_uint64)]

    g = Guarded()
    g.guard = 0x0123456789ABCDEF
    n = ctypes.c_int32(0)
    geom = pkv._geom(b1.B, b1.Hq, b1.Hkv, b1.D, b1.max_pages, b1.num_pages)
    opts = pkv._opts(num_sms=NUM_SMS)
    rc = lib.pkv_plan_dry_run(lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), None, 16, ctypes.byref(geom),
                              ctypes.byref(opts), ctypes.byref(g.info), None, 0, ctypes.byref(n))
    assert rc == 0 and g.guard == 0x0123456789ABCDEF
    assert g.info.copy in (pkv.COPY["lsu"], pkv.COPY["tma"]) and g.info.kv_bytes == 4096 * 8 * 128 * 4


def test_splits_are_capped_by_the_merge_scratch():
    p = _geom_problem([4096 * 16], Hq=8, Hkv=1, D=64)   # G = 8: at most 4096 / 8 splits
    info, q = _dry(p, force_mode="split_queue", num_splits=5000)
    assert info["max_splits"] <= 512


@pytest.mark.parametrize("bad,code", [
    (dict(Hq=6, Hkv=4), pkv.EINVAL),          # G not an integer
    (dict(D=96), pkv.EUNSUPPORTED),           # head dim without kernels
    (dict(Hq=32, Hkv=2), pkv.EUNSUPPORTED),   # G = 16
    (dict(ps=8), pkv.EUNSUPPORTED),           # page not a multiple of 16
])
def test_geometry_errors(bad, code):
    kw = dict(Hq=8, Hkv=2, D=64, ps=16)
    kw.update(bad)
    lens = np.array([20, 40], np.int32)
    with pytest.raises(pkv.PkvError) as e:
        pkv.dry_run(lens, None, kw["ps"], B=2, Hq=kw["Hq"], Hkv=kw["Hkv"], D=kw["D"], max_pages=8,
                    num_pages=16, num_sms=NUM_SMS)
    assert e.value.code == code


def test_row_errors():
    p = _geom_problem([20, 40])
    with pytest.raises(pkv.PkvError) as e:   # longer than the table row allows
        pkv.dry_run([20, 16 * p.max_pages + 1], None, 16, B=2, Hq=8, Hkv=2, D=64, max_pages=p.max_pages,
                    num_pages=p.num_pages, num_sms=NUM_SMS)
    assert e.value.code == pkv.EINVAL
    with pytest.raises(pkv.PkvError):        # negative length
        pkv.dry_run([-1, 4], None, 16, B=2, Hq=8, Hkv=2, D=64, max_pages=4, num_pages=16, num_sms=NUM_SMS)
    bad = p.block_table.copy()
    bad[1, 2] = p.num_pages                   # page id out of the pool
    with pytest.raises(pkv.PkvError):
        pkv.dry_run(p.seq_lens, bad, 16, B=2, Hq=8, Hkv=2, D=64, max_pages=p.max_pages,
                    num_pages=p.num_pages, num_sms=NUM_SMS)
    with pytest.raises(pkv.PkvError):        # no SM count and no device to ask
        pkv.dry_run(p.seq_lens, None, 16, B=2, Hq=8, Hkv=2, D=64, max_pages=p.max_pages,
                    num_pages=p.num_pages)
    with pytest.raises(pkv.PkvError):        # unknown mode
        pkv.dry_run(p.seq_lens, None, 16, B=2, Hq=8, Hkv=2, D=64, max_pages=p.max_pages,
                    num_pages=p.num_pages, num_sms=NUM_SMS, force_mode=9)


def test_pool_reserve_and_release():
    pool = pkv.Pool([7, 3, 9, 1], num_pages=10)
    table = np.full((3, 4), -1, np.int32)
    table[0, 0] = 5
    table[1, :2] = [6, 8]
    lens = np.array([16, 20, 0], np.int32)   # row 0 at a page boundary, row 1 mid-page, row 2 empty
    rows = pool.reserve(lens, table, 16)
    assert rows.tolist() == [0, 2]
    assert table[0].tolist() == [5, 7, -1, -1] and table[2].tolist() == [3, -1, -1, -1]
    assert table[1].tolist() == [6, 8, -1, -1]
    assert pool.free_count() == 2
    assert pool.reserve(lens, table, 16).tolist() == []   # entries already assigned: nothing to do
    pool.release([7])
    assert pool.free_count() == 3


def test_pool_exhaustion_changes_nothing():
    pool = pkv.Pool([4], num_pages=8)
    table = np.full((2, 2), -1, np.int32)
    before = table.copy()
    with pytest.raises(pkv.PkvError) as e:
        pool.reserve(np.array([0, 0], np.int32), table, 16)
    assert e.value.code == pkv.ENOSPACE
    assert np.array_equal(table, before) and pool.free_count() == 1
    full = np.zeros((1, 2), np.int32)
    with pytest.raises(pkv.PkvError) as e:     # row already holds max_pages pages
        pool.reserve(np.array([32], np.int32), full, 16)
    assert e.value.code == pkv.ENOSPACE
    with pytest.raises(pkv.PkvError):
        pkv.Pool([8], num_pages=8)             # page id outside the pool


def test_pool_refuses_a_page_twice():
    with pytest.raises(pkv.PkvError) as e:
        pkv.Pool([2, 5, 2], num_pages=8)       # listed twice
    assert e.value.code == pkv.EINVAL
    pool = pkv.Pool([2, 5], num_pages=8)
    for again in ([5], [6, 2], [6, 6]):        # already free, or twice in one call
        with pytest.raises(pkv.PkvError) as e:
            pool.release(again)
        assert e.value.code == pkv.EINVAL
        assert pool.free_count() == 2          # nothing changed
    table = np.full((1, 2), -1, np.int32)
    pool.reserve(np.array([0], np.int32), table, 16)
    assert table[0, 0] == 2 and pool.free_count() == 1
    pool.release([2, 6])                       # 2 is in use again, 6 never was free: both come back
    assert pool.free_count() == 3
    with pytest.raises(pkv.PkvError):
        pool.release([2])


def test_strerror_covers_every_code():
    lib = pkv.load()
    for code in range(7):
        assert lib.pkv_strerror(code).decode() not in ("", "unknown error")
    assert lib.pkv_strerror(99).decode() == "unknown error"


@pytest.mark.parametrize("kind", ["uniform", "bimodal", "zipf", "bucketed"])
def test_trace_lengths_follow_their_recipes(kind):
    rng = np.random.default_rng(wl.CALIBRATION_SEED)
    n = wl.trace_lengths(kind, 4000, rng)
    assert n.dtype == np.int32 and n.min() >= 256 and n.max() <= 32768
    if kind == "uniform":
        assert n.min() >= 512 and abs(n.mean() - (512 + 32768) / 2) < 600
    elif kind == "bimodal":
        short, long_ = n[n <= 2048], n[n >= 16384]
        assert len(short) + len(long_) == len(n) and abs(len(short) / len(n) - 0.5) < 0.05
    elif kind == "zipf":
        from scipy.special import zeta
        assert np.all(n % 512 == 0) and n.max() == 32768
        assert abs(np.mean(n == 512) - 1 / zeta(1.3)) < 0.02   # P(k = 1) of Zipf(1.3)
    else:
        assert set(n.tolist()) == {1024, 4096, 16384, 32768}
    again = wl.trace_lengths(kind, 4000, np.random.default_rng(wl.CALIBRATION_SEED))
    assert np.array_equal(n, again)


def test_policy_on_trace_families_never_picks_direct_below_one_wave():
    for kind in ["uniform", "bimodal", "zipf", "bucketed"]:
        for B in (1, 4, 8):
            lens = wl.trace_lengths(kind, B, np.random.default_rng(wl.HELD_OUT_SEED))
            p = _geom_problem(lens, Hq=32, Hkv=8, D=128)
            info, q = _dry(p)
            if max(lens) > 16 * 8:
                assert info["mode_name"] == "split_queue", (kind, B)
                assert info["num_work_items"] <= 2 * NUM_SMS


def test_merge_choice_follows_route_and_wave():
    """Fused merge: the last arriving split merges (LAST) unless every split is asked
    to share it out (ALL), which needs a split launch of one wave of resident CTAs.
    The dry run takes num_sms * ctas_per_sm as the resident capacity."""
    lens = [4096, 1000, 17, 0]
    kw = dict(B=4, Hq=8, Hkv=2, D=128, max_pages=256, num_pages=600)

    def info(**o):
        return pkv.dry_run(lens, None, 16, num_sms=NUM_SMS, ctas_per_sm=2, **kw, **o)[0]

    assert info(force_mode="split_queue", num_splits=8)["merge_name"] == "last"
    assert info(force_mode="split_queue", num_splits=8, merge="all")["merge_name"] == "all"
    assert info(force_mode="split_padded", num_splits=8, merge="all")["merge_name"] == "all"
    assert info(force_mode="split_queue", num_splits=8, merge="last")["merge_name"] == "last"
    assert info(force_mode="split_queue", num_splits=8, separate_merge=True)["merge_name"] == "separate"
    assert info(force_mode="persistent", num_splits=8)["merge_name"] == "last"
    assert info(force_mode="direct")["merge_name"] == "none"
    assert info(force_mode="split_queue", num_splits=1)["merge_name"] == "none"
    # more tiles than resident CTAs: ALL is refused
    small = dict(num_sms=4, ctas_per_sm=2)
    i = pkv.dry_run(lens, None, 16, **small, **kw, force_mode="split_queue", num_splits=8)[0]
    assert i["num_tiles"] > 8 and i["merge_name"] == "last"
    with pytest.raises(pkv.PkvError) as e:
        pkv.dry_run(lens, None, 16, **small, **kw, force_mode="split_queue", num_splits=8, merge="all")
    assert e.value.code == pkv.EUNSUPPORTED
