"""Pins for the oracle's slot model (oracle/slots.py): the FIFO page rule with
slot admit / evict, checked against a hand-worked example and against
invariants (every page is free or in exactly one table; prompts land where the
paged layout puts them)."""
import numpy as np

from oracle.slots import SlotModel, write_prompt


def test_hand_worked_sequence():
    """page_size 2, three rows, max 4 pages; free list [3, 0, 6, 2, 4].
    step 1: row 1's next token (position 2) has page 7 already; row 2 (length 0)
            takes 3 -> lens [2, 3, 1], free [0, 6, 2, 4]
    evict [1]: pages 1, 7 to the back -> free [0, 6, 2, 4, 1, 7]
    admit [1] with 3 tokens: pages 0, 6 -> free [2, 4, 1, 7]
    step 2: row 0 (position 2) takes 2 -> lens [3, 4, 2], free [4, 1, 7]
    evict [2, 0]: 3, then 5, 2 -> free [4, 1, 7, 3, 5, 2]
    step 3: only row 1 is active; position 4 takes 4 -> lens [0, 5, 0], free [1, 7, 3, 5, 2]"""
    table = np.full((3, 4), -1, np.int32)
    table[0, 0] = 5
    table[1, :2] = [1, 7]
    m = SlotModel([1, 2, 0], table, [3, 0, 6, 2, 4], 2)
    m.step(None, None)
    assert m.lens.tolist() == [2, 3, 1] and list(m.free) == [0, 6, 2, 4] and m.table[2, 0] == 3
    m.evict([1])
    assert list(m.free) == [0, 6, 2, 4, 1, 7] and m.table[1].tolist() == [-1] * 4 and m.lens[1] == 0
    m.admit([1], [3])
    assert m.table[1].tolist() == [0, 6, -1, -1] and m.lens[1] == 3 and list(m.free) == [2, 4, 1, 7]
    m.step(None, None)
    assert m.lens.tolist() == [3, 4, 2] and m.table[0].tolist() == [5, 2, -1, -1] and list(m.free) == [4, 1, 7]
    m.evict([2, 0])
    assert list(m.free) == [4, 1, 7, 3, 5, 2] and m.active.tolist() == [0, 1, 0]
    m.step(None, None)
    assert m.lens.tolist() == [0, 5, 0] and m.table[1].tolist() == [0, 6, 4, -1]
    assert list(m.free) == [1, 7, 3, 5, 2]


def test_pages_are_conserved_and_prompts_land_in_place():
    rng = np.random.default_rng(7)
    ps, NP, B, mp, Hkv, D = 4, 64, 5, 12, 2, 8
    k = rng.integers(0, 65535, size=(NP, ps, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 65535, size=(NP, ps, Hkv, D), dtype=np.uint16)
    lens = [3, 8, 0, 5, 1]
    perm = rng.permutation(NP).astype(np.int32)
    table = np.full((B, mp), -1, np.int32)
    at = 0
    for b, n in enumerate(lens):
        p = -(-n // ps)
        table[b, :p] = perm[at:at + p]
        at += p
    m = SlotModel(lens, table, perm[at:], ps, k, v)
    for step in range(20):
        if step == 5:
            m.evict([1, 4])
        if step == 9:
            n = [9, 4]
            ks = rng.integers(0, 65535, size=(sum(n), Hkv, D), dtype=np.uint16)
            vs = rng.integers(0, 65535, size=(sum(n), Hkv, D), dtype=np.uint16)
            m.admit([4, 1], n, ks, vs)
            # the prompts read back through the table, token by token
            for (b, lo, hi) in ((4, 0, 9), (1, 9, 13)):
                for t in range(hi - lo):
                    page = m.table[b, t // ps]
                    assert np.array_equal(m.k_pages[page, t % ps], ks[lo + t])
                    assert np.array_equal(m.v_pages[page, t % ps], vs[lo + t])
        kn = rng.integers(0, 65535, size=(B, Hkv, D), dtype=np.uint16)
        m.step(kn, kn)
        used = [int(x) for x in m.table.ravel() if x >= 0]
        assert len(used) == len(set(used))
        assert sorted(used + list(m.free)) == list(range(NP))
        for b in range(B):   # pages cover exactly the tokens of an active row
            assert (m.table[b] >= 0).sum() == -(-int(m.lens[b]) // ps)


def test_write_prompt_follows_the_layout():
    k = np.zeros((6, 4, 1, 2), np.uint16)
    v = np.zeros_like(k)
    src = np.arange(7 * 2, dtype=np.uint16).reshape(7, 1, 2) + 1
    write_prompt(src, src + 100, k, v, np.array([4, 1, -1]), 7)
    assert k[4, 0, 0].tolist() == [1, 2] and k[4, 3, 0].tolist() == [7, 8]
    assert k[1, 0, 0].tolist() == [9, 10] and k[1, 2, 0].tolist() == [13, 14] and k[1, 3, 0].tolist() == [0, 0]
    assert v[1, 2, 0].tolist() == [113, 114]
