"""Pins for the oracle's work-tile enumeration and KV append.

The queue rule is the reading stated in oracle/queue.py of "PersistentKV"
(gist.science summary), Methodology section 1 ("Sequence Splitting",
"Row-Local Bounds", "Compact Workqueue").
"""
import os

import numpy as np
import pytest

import oracle
from paged_kv_decode_block_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_queues():
    """{S: tiles} of the split queues and {"direct": tiles} of the single-pass route."""
    out = {}
    for line in open(os.path.join(GOLDEN, "tiny_queue.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        key, *tile = line.split()
        out.setdefault(key if key == "direct" else int(key), []).append(list(map(int, tile)))
    return out


@pytest.mark.parametrize("S", [1, 2, 4])
def test_tiny_queue_matches_hand_derivation(S):
    p = wl.tiny()
    C = oracle.chunk_pages_for_splits(p.seq_lens, p.page_size, S)
    got = oracle.enumerate_queue(p.seq_lens, p.page_size, p.Hkv, C)
    assert got.tolist() == _golden_queues()[S]


def test_tiny_direct_tiles_match_hand_derivation():
    p = wl.tiny()
    got = oracle.enumerate_direct(p.seq_lens, p.page_size, p.Hkv)
    assert got.tolist() == _golden_queues()["direct"]


@pytest.mark.parametrize("seed", range(4))
def test_direct_tiles_cover_every_row_once(seed):
    """One tile per (b, kvh) in (b, kvh) order, split 0, pages [0, P_b) with P_b
    counted by brute force over the tokens; empty rows keep their (empty) tile."""
    rng = np.random.default_rng(100 + seed)
    B, Hkv, ps = int(rng.integers(1, 7)), int(rng.integers(1, 5)), int(rng.choice([1, 16, 64]))
    lens = rng.integers(0, 300, size=B)
    lens[0] = 0
    d = oracle.enumerate_direct(lens, ps, Hkv)
    assert d.shape == (B * Hkv, 5)
    i = 0
    for b, n in enumerate(lens):
        pages = len({t // ps for t in range(int(n))})
        for kvh in range(Hkv):
            assert d[i].tolist() == [b, kvh, 0, 0, pages]
            i += 1
    # with one chunk covering every row, the compact queue is the direct list minus empty rows
    C = max(1, int(d[:, 4].max()))
    q = oracle.enumerate_queue(lens, ps, Hkv, C)
    assert q.tolist() == d[d[:, 4] > 0].tolist()


def _check_queue_properties(lens, ps, Hkv, C):
    q = oracle.enumerate_queue(lens, ps, Hkv, C)
    # strictly increasing (b, kvh, s): lexicographic order, no duplicates
    keys = [tuple(t[:3]) for t in q]
    assert keys == sorted(keys) and len(set(keys)) == len(keys)
    # no empty tile, at most C pages each
    assert np.all(q[:, 4] > q[:, 3]) if len(q) else True
    assert np.all(q[:, 4] - q[:, 3] <= C) if len(q) else True
    # per (b, kvh) the tiles tile [0, P_b) exactly, in order, brute force over pages
    for b, n in enumerate(lens):
        P = -(-int(n) // ps)
        for kvh in range(Hkv):
            covered = []
            for t in q[(q[:, 0] == b) & (q[:, 1] == kvh)]:
                covered.extend(range(t[3], t[4]))
            assert covered == list(range(P))
    expected = Hkv * sum(-(-(-(-int(n) // ps)) // C) for n in lens)
    assert len(q) == expected
    # the padded grid holds the same non-empty tiles plus empty slots for s >= S_b
    grid = oracle.enumerate_padded_grid(lens, ps, Hkv, C)
    nonempty = grid[grid[:, 4] > grid[:, 3]]
    assert nonempty.tolist() == q.tolist()
    s_max = -(-max((-(-int(n) // ps) for n in lens), default=0) // C)
    assert len(grid) == len(lens) * Hkv * s_max


@pytest.mark.parametrize("seed", range(6))
def test_queue_properties_random(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 9))
    lens = rng.integers(0, 400, size=B)
    ps = int(rng.choice([1, 4, 16]))
    Hkv = int(rng.integers(1, 4))
    C = int(rng.integers(1, 12))
    _check_queue_properties(lens, ps, Hkv, C)


def test_queue_batch1_long_shape():
    """32768 tokens in 16-token pages with 32 splits: 64-page chunks, 8 x 32 tiles."""
    lens = [32768]
    C = oracle.chunk_pages_for_splits(lens, 16, 32)
    assert C == 64
    q = oracle.enumerate_queue(lens, 16, 8, C)
    assert q.shape == (256, 5)
    assert q[-1].tolist() == [0, 7, 31, 1984, 2048]


def test_append_places_bytes_and_bumps_lengths():
    p = wl.make_problem("append", [15, 16, 0], Hq=4, Hkv=2, D=8, page_size=16, num_pages=8,
                        max_pages=2, seed=3)
    table = p.block_table.copy()
    table[1, 1] = p.free_pages[0]   # row 1 is at a page boundary: give it its next page
    table[2, 0] = p.free_pages[1]
    rng = np.random.default_rng(4)
    kn, vn = wl.new_tokens(rng, 3, 2, 8)
    k2, v2, lens2 = oracle.append(kn, vn, p.k_pages, p.v_pages, table, p.seq_lens)
    assert lens2.tolist() == [16, 17, 1]
    assert np.array_equal(k2[table[0, 0], 15], kn[0]) and np.array_equal(v2[table[0, 0], 15], vn[0])
    assert np.array_equal(k2[table[1, 1], 0], kn[1]) and np.array_equal(v2[table[1, 1], 0], vn[1])
    assert np.array_equal(k2[table[2, 0], 0], kn[2])
    changed = np.argwhere(np.any(k2 != p.k_pages, axis=(2, 3)))
    assert len(changed) <= 3   # nothing else moved


def test_append_then_decode_sees_new_token():
    """Decoding after an append equals decoding a problem built with that token in place."""
    p = wl.make_problem("append2", [20, 31], Hq=4, Hkv=1, D=16, page_size=8, num_pages=10,
                        max_pages=5, seed=5)
    rng = np.random.default_rng(6)
    kn, vn = wl.new_tokens(rng, 2, 1, 16)
    k2, v2, lens2 = oracle.append(kn, vn, p.k_pages, p.v_pages, p.block_table, p.seq_lens)
    out_a, lse_a = oracle.decode(p.q, k2, v2, p.block_table, lens2)
    k3, v3 = p.k_pages.copy(), p.v_pages.copy()
    for b in range(2):
        n = int(p.seq_lens[b])
        page = p.block_table[b, n // 8]
        k3[page, n % 8] = kn[b]
        v3[page, n % 8] = vn[b]
    out_b, lse_b = oracle.decode(p.q, k3, v3, p.block_table, p.seq_lens + 1)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_append_rejects_full_row():
    p = wl.make_problem("full", [32], Hq=1, Hkv=1, D=8, page_size=16, num_pages=2, seed=1)
    kn, vn = wl.new_tokens(np.random.default_rng(0), 1, 1, 8)
    with pytest.raises(ValueError):
        oracle.append(kn, vn, p.k_pages, p.v_pages, p.block_table, p.seq_lens)


def test_append_in_place_equals_copying_append():
    p = wl.make_problem("inplace", [15, 16, 3], Hq=2, Hkv=1, D=8, page_size=16, num_pages=6,
                        max_pages=2, seed=9)
    table = p.block_table.copy()
    table[1, 1] = p.free_pages[0]
    kn, vn = wl.new_tokens(np.random.default_rng(10), 3, 1, 8)
    k2, v2, l2 = oracle.append(kn, vn, p.k_pages, p.v_pages, table, p.seq_lens)
    k3, v3, l3 = p.k_pages.copy(), p.v_pages.copy(), p.seq_lens.copy()
    r = oracle.append(kn, vn, k3, v3, table, l3, inplace=True)
    assert r[0] is k3 and r[1] is v3 and r[2] is l3
    assert np.array_equal(k2, k3) and np.array_equal(v2, v3) and np.array_equal(l2, l3)
