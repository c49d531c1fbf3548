"""pkv_append through the C ABI on the GPU, with its failure flags.

The append writes row b's new K/V token at position seq_lens[b] (page
block_table[b][pos / page_size], slot pos % page_size) and then increments the
length ("PersistentKV" gist.science summary, Methodology section 1 "Layout";
the KV-cache update operator of "GPUOS", arXiv 2604.17861, section 4).  A row
with no page for its new token (table full, or the entry unassigned) must set
PKV_DEV_ROW_FULL, and one whose entry names a page past the pool must set
PKV_DEV_PAGE_OOB; in both cases the kernel checks before any access, writes no
page byte for that row and leaves its length as it was.  The good rows are
checked bit for bit against the oracle's append.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl
from pkv_testutil import make_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load()


def _problem():
    # rows: 0 and 1 ordinary (1 ends mid-page), 2 at a page boundary with an
    # unassigned entry, 3 with its table full, 4 whose next entry names a page
    # past the pool; max_pages 4 for every row
    lens = [20, 33, 32, 64, 47]
    p = wl.make_problem("append_flags", lens, Hq=8, Hkv=2, D=64, page_size=16, num_pages=24,
                        max_pages=4, seed=53)
    table = p.block_table.copy()
    assert table[2, 2] == -1 and table[3, 3] >= 0
    table[4, 2] = p.num_pages + 5   # past the pool: the row's page of position 47
    return p, table


def _run_append(p, table, kn, vn):
    dev_k = torch.from_numpy(p.k_pages.view(np.int16)).cuda()
    dev_v = torch.from_numpy(p.v_pages.view(np.int16)).cuda()
    dev_t = torch.from_numpy(table).cuda()
    dev_l = torch.from_numpy(p.seq_lens.copy()).cuda()
    plan = make_plan(p, host_table=False, force_mode="direct")
    pkv.append(torch.from_numpy(kn.view(np.int16)).cuda(), torch.from_numpy(vn.view(np.int16)).cuda(),
               dev_k, dev_v, dev_t, dev_l, plan)
    torch.cuda.synchronize()
    status = plan.status()
    return (dev_k.cpu().numpy().view(np.uint16), dev_v.cpu().numpy().view(np.uint16), dev_l.cpu().numpy(),
            dev_t.cpu().numpy(), status)


def test_append_flags_rows_without_a_valid_page_and_leaves_them_unchanged():
    p, table = _problem()
    rng = np.random.default_rng(54)
    kn, vn = wl.new_tokens(rng, p.B, p.Hkv, p.D)
    k, v, lens, table_after, status = _run_append(p, table, kn, vn)
    assert status & pkv.DEV_ROW_FULL and status & pkv.DEV_PAGE_OOB
    assert np.array_equal(table_after, table)
    good = [0, 1]
    bad = [2, 3, 4]
    assert lens[good].tolist() == [21, 34]
    assert lens[bad].tolist() == p.seq_lens[bad].tolist()
    # expected pools: the oracle's append of the good rows only
    sub = np.array(good)
    k_ref, v_ref, _ = oracle.append(kn[sub], vn[sub], p.k_pages, p.v_pages, table[sub], p.seq_lens[sub])
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_append_of_good_rows_sets_no_flag():
    p, table = _problem()
    sub = [0, 1]
    q = wl.make_problem("append_ok", p.seq_lens[sub], Hq=8, Hkv=2, D=64, page_size=16, num_pages=24,
                        max_pages=4, seed=55)
    rng = np.random.default_rng(56)
    kn, vn = wl.new_tokens(rng, q.B, q.Hkv, q.D)
    k, v, lens, _, status = _run_append(q, q.block_table.copy(), kn, vn)
    assert status == 0
    k_ref, v_ref, l_ref = oracle.append(kn, vn, q.k_pages, q.v_pages, q.block_table, q.seq_lens)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref) and np.array_equal(lens, l_ref)
