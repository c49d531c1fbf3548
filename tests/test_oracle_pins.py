"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an oracle library handle and raises AssertionError
on a mismatch.  The tests run them on the real oracle; ``test_pins_catch_planted_mistakes``
runs them on copies of the oracle with a mistake planted in the C source, and
requires every mutant to be caught by at least one pin.

Reading pinned throughout: scaled dot-product attention of one query token per
head (scale 1/sqrt(D), natural-log LSE), query head h reading KV head floor(h/G),
token t of row b at page block_table[b][t // ps], slot t % ps -- "PersistentKV:
Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs"
(gist.science summary), Technical Summary, Methodology section 1.
"""
import json
import math
import os
import shutil

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_decode_block_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAN_BF16 = 0x7FC0


# --- helpers ---------------------------------------------------------------------------

def _contiguous_problem(rng, B, Hq, Hkv, D, ps, lens):
    """Rows own consecutive physical pages (identity-like table), random bf16 data."""
    lens = np.asarray(lens, np.int32)
    max_pages = max(1, max(-(-int(n) // ps) for n in lens))
    NP = B * max_pages
    table = np.arange(NP, dtype=np.int32).reshape(B, max_pages)
    q = wl.bf16_normal(rng, (B, Hq, D))
    k = wl.bf16_normal(rng, (NP, ps, Hkv, D))
    v = wl.bf16_normal(rng, (NP, ps, Hkv, D))
    return q, k, v, table, lens


def _dense_rows(k_pages, table, b, n):
    """K (or V) of row b as a dense [n][Hkv][D] float64 array, for a contiguous table."""
    NP, ps, Hkv, D = k_pages.shape
    pages = k_pages[table[b, : -(-n // ps)]] if n else k_pages[:0]
    return wl.bf16_to_float32(pages.reshape(-1, Hkv, D)[:n]).astype(np.float64)


def _library_attention(q, k_pages, v_pages, table, lens):
    """Attention through torch's CPU attention kernels in float64 (library routine):
    the flash-attention CPU op gives out and logsumexp; SDPA with enable_gqa gives
    out again with torch's own GQA head grouping."""
    B, Hq, D = q.shape
    Hkv = k_pages.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    for b in range(B):
        n = int(lens[b])
        qt = torch.from_numpy(wl.bf16_to_float32(q[b]).astype(np.float64)).reshape(1, Hq, 1, D)
        kt = torch.from_numpy(_dense_rows(k_pages, table, b, n)).permute(1, 0, 2).unsqueeze(0)
        vt = torch.from_numpy(_dense_rows(v_pages, table, b, n)).permute(1, 0, 2).unsqueeze(0)
        o_gqa = F.scaled_dot_product_attention(qt, kt, vt, enable_gqa=True)
        o, l = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
            qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1), 0.0, False)[:2]
        assert torch.allclose(o, o_gqa, atol=1e-13, rtol=0)
        out[b] = o.reshape(Hq, D).numpy()
        lse[b] = l.reshape(Hq).numpy()
    return out, lse


def _from_json_array(x, shape):
    """Nested lists of numbers of the given shape; the string "NaN" stands for a whole
    NaN sub-array at whatever level it appears."""
    if isinstance(x, str):
        assert x == "NaN"
        return np.full(shape, np.float32("nan"), np.float32)
    if not shape:
        return np.float32(x)
    assert len(x) == shape[0]
    return np.stack([_from_json_array(e, shape[1:]) for e in x])


def _golden_case(case):
    q = np.array(case["q"], np.float32)
    B, Hq, D = q.shape
    k_raw = case["k_pages"]
    NP, ps = len(k_raw), case["page_size"]
    # Hkv from the first slot that is spelled out
    hkv = next(len(s) for p in k_raw if not isinstance(p, str) for s in p if not isinstance(s, str))
    shape = (NP, ps, hkv, D)

    def build(raw):
        arr = _from_json_array(raw, shape)
        bits = wl.round_to_bf16(np.nan_to_num(arr, nan=0.0))
        bits[np.isnan(arr)] = NAN_BF16
        assert np.array_equal(wl.bf16_to_float32(bits)[~np.isnan(arr)], arr[~np.isnan(arr)]), \
            "golden inputs must be exact in bf16"
        return bits

    env = {"e": math.e, "ln": math.log, "inf": math.inf}
    ev = np.vectorize(lambda s: float(eval(s, {"__builtins__": {}}, env)), otypes=[np.float64])
    return dict(q=wl.round_to_bf16(q), k=build(case["k_pages"]), v=build(case["v_pages"]),
                table=np.array(case["block_table"], np.int32),
                lens=np.array(case["seq_lens"], np.int32),
                out=ev(np.array(case["expected_out"], dtype=object)),
                lse=ev(np.array(case["expected_lse"], dtype=object)).reshape(B, Hq))


# --- pins ------------------------------------------------------------------------------

def pin_golden(lib):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        c = _golden_case(case)
        out, lse = oracle.decode(c["q"], c["k"], c["v"], c["table"], c["lens"], lib=lib)
        assert np.allclose(out, c["out"], atol=1e-14, rtol=0), case["name"]
        assert np.array_equal(np.isneginf(lse), np.isneginf(c["lse"])), case["name"]
        fin = np.isfinite(c["lse"])
        assert np.allclose(lse[fin], c["lse"][fin], atol=1e-14, rtol=0), case["name"]


LIB_SHAPES = [  # B, Hq, Hkv, D, ps, lens
    (1, 1, 1, 8, 4, [1]),
    (2, 4, 1, 64, 16, [37, 100]),
    (3, 8, 2, 16, 8, [8, 9, 23]),
    (2, 8, 8, 32, 16, [16, 17]),
    (1, 16, 2, 128, 16, [300]),
]


def pin_library_attention(lib):
    rng = np.random.default_rng(7)
    for B, Hq, Hkv, D, ps, lens in LIB_SHAPES:
        q, k, v, table, lens = _contiguous_problem(rng, B, Hq, Hkv, D, ps, lens)
        out, lse = oracle.decode(q, k, v, table, lens, lib=lib)
        ref_out, ref_lse = _library_attention(q, k, v, table, lens)
        assert np.allclose(out, ref_out, atol=1e-12, rtol=0), (B, Hq, Hkv, D, ps)
        assert np.allclose(lse, ref_lse, atol=1e-12, rtol=0), (B, Hq, Hkv, D, ps)


def pin_one_token(lib):
    rng = np.random.default_rng(11)
    q, k, v, table, lens = _contiguous_problem(rng, 2, 4, 2, 16, 4, [1, 1])
    out, lse = oracle.decode(q, k, v, table, lens, lib=lib)
    for b in range(2):
        for h in range(4):
            v0 = _dense_rows(v, table, b, 1)[0, h // 2]
            assert np.array_equal(out[b, h], v0)
            k0 = torch.from_numpy(_dense_rows(k, table, b, 1)[0, h // 2])
            q0 = torch.from_numpy(wl.bf16_to_float32(q[b, h]).astype(np.float64))
            assert math.isclose(lse[b, h], float(torch.dot(q0, k0)) / 4.0, rel_tol=1e-15, abs_tol=1e-15)


def pin_constant_v(lib):
    rng = np.random.default_rng(12)
    q, k, v, table, lens = _contiguous_problem(rng, 2, 8, 2, 32, 16, [45, 130])
    c = wl.bf16_normal(rng, (2, 32))  # one constant vector per KV head
    v[:] = c[None, None, :, :]
    out, _ = oracle.decode(q, k, v, table, lens, lib=lib)
    want = wl.bf16_to_float32(c).astype(np.float64)
    for h in range(8):
        assert np.allclose(out[:, h], want[h // 4], atol=1e-14, rtol=0)


def pin_zero_query(lib):
    rng = np.random.default_rng(13)
    q, k, v, table, lens = _contiguous_problem(rng, 2, 4, 2, 16, 8, [5, 29])
    q[:] = 0
    out, lse = oracle.decode(q, k, v, table, lens, lib=lib)
    for b in range(2):
        n = int(lens[b])
        vm = _dense_rows(v, table, b, n).mean(axis=0)
        for h in range(4):
            assert np.allclose(out[b, h], vm[h // 2], atol=1e-14, rtol=0)
            assert math.isclose(lse[b, h], math.log(n), rel_tol=0, abs_tol=1e-14)


def pin_gqa_mapping(lib):
    """Only KV head j carries non-zero V: exactly the query heads floor(h/G) == j see it."""
    rng = np.random.default_rng(14)
    B, Hq, Hkv = 1, 8, 4
    q, k, v, table, lens = _contiguous_problem(rng, B, Hq, Hkv, 8, 4, [10])
    for j in range(Hkv):
        vj = v.copy()
        vj[:, :, [i for i in range(Hkv) if i != j], :] = 0
        out, _ = oracle.decode(q, k, vj, table, lens, lib=lib)
        for h in range(Hq):
            nonzero = bool(np.any(out[0, h] != 0))
            assert nonzero == (h // (Hq // Hkv) == j), (j, h)


def pin_block_table_permutation(lib):
    """Moving pages to other physical slots (data moved with them) changes nothing."""
    p = wl.tiny()
    out0, lse0 = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, lib=lib)
    rng = np.random.default_rng(15)
    perm = rng.permutation(p.num_pages)          # new physical slot of each page
    k2 = np.empty_like(p.k_pages)
    v2 = np.empty_like(p.v_pages)
    k2[perm] = p.k_pages
    v2[perm] = p.v_pages
    table2 = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    out1, lse1 = oracle.decode(p.q, k2, v2, table2, p.seq_lens, lib=lib)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_tokens_past_length_unread(lib):
    """NaN in slots past N_b and in pages no row owns leaves the result untouched."""
    p = wl.tiny()
    out0, lse0 = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, lib=lib)
    k, v = p.k_pages.copy(), p.v_pages.copy()
    used = set()
    for b, n in enumerate(p.seq_lens):
        P = -(-int(n) // p.page_size)
        used.update(int(x) for x in p.block_table[b, :P])
        last = int(p.block_table[b, P - 1])
        k[last, int(n) - (P - 1) * p.page_size:] = NAN_BF16
        v[last, int(n) - (P - 1) * p.page_size:] = NAN_BF16
    for page in set(range(p.num_pages)) - used:
        k[page] = NAN_BF16
        v[page] = NAN_BF16
    out1, lse1 = oracle.decode(p.q, k, v, p.block_table, p.seq_lens, lib=lib)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def _split_and_merge(p, num_splits, lib):
    C = oracle.chunk_pages_for_splits(p.seq_lens, p.page_size, num_splits)
    tiles = oracle.enumerate_queue(p.seq_lens, p.page_size, p.Hkv, C)
    G = p.Hq // p.Hkv
    parts = {}
    for b, kvh, s, pb, pe in tiles:
        o, l = oracle.partial(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, b, kvh,
                              pb * p.page_size, pe * p.page_size, lib=lib)
        parts.setdefault((b, kvh), []).append((o, l))
    out = np.zeros((p.B, p.Hq, p.D))
    lse = np.full((p.B, p.Hq), -np.inf)
    for (b, kvh), lst in parts.items():
        for g in range(G):
            o_s = np.stack([o[g] for o, _ in lst])
            l_s = np.array([l[g] for _, l in lst])
            out[b, kvh * G + g], lse[b, kvh * G + g] = oracle.merge(o_s, l_s, lib=lib)
    return out, lse


def pin_split_merge_equals_unsplit(lib):
    probs = [wl.tiny(),
             wl.make_problem("ragged", [1, 16, 17, 95, 0], Hq=6, Hkv=3, D=16, page_size=8,
                             num_pages=40, seed=16)]
    for p in probs:
        out0, lse0 = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, lib=lib)
        p_max = max(-(-int(n) // p.page_size) for n in p.seq_lens)
        for S in range(1, p_max + 1):
            out1, lse1 = _split_and_merge(p, S, lib)
            assert np.allclose(out1, out0, atol=1e-12, rtol=0), (p.name, S)
            assert np.array_equal(np.isneginf(lse0), np.isneginf(lse1))
            fin = np.isfinite(lse0)
            assert np.allclose(lse1[fin], lse0[fin], atol=1e-12, rtol=0), (p.name, S)


def pin_merge_identities(lib):
    rng = np.random.default_rng(17)
    o = rng.standard_normal((3, 8))
    l = rng.standard_normal(3) * 4
    one, one_l = oracle.merge(o[:1], l[:1], lib=lib)
    assert np.array_equal(one, o[0]) and one_l == l[0]
    with_neutral, wl_ = oracle.merge(np.vstack([o, np.zeros((1, 8))]), np.append(l, -np.inf), lib=lib)
    base, base_l = oracle.merge(o, l, lib=lib)
    assert np.allclose(with_neutral, base, atol=1e-15) and math.isclose(wl_, base_l, abs_tol=1e-15)
    rev, rev_l = oracle.merge(o[::-1], l[::-1], lib=lib)
    assert np.allclose(rev, base, atol=1e-14) and math.isclose(rev_l, base_l, abs_tol=1e-14)
    # two equal halves: lse grows by ln 2, the output is unchanged
    two, two_l = oracle.merge(np.vstack([o[0], o[0]]), np.array([l[0], l[0]]), lib=lib)
    assert np.allclose(two, o[0], atol=1e-15) and math.isclose(two_l, l[0] + math.log(2), abs_tol=1e-14)
    empty, empty_l = oracle.merge(np.zeros((2, 8)), np.array([-np.inf, -np.inf]), lib=lib)
    assert np.array_equal(empty, np.zeros(8)) and empty_l == -np.inf


ALL_PINS = [pin_golden, pin_library_attention, pin_one_token, pin_constant_v, pin_zero_query,
            pin_gqa_mapping, pin_block_table_permutation, pin_tokens_past_length_unread,
            pin_split_merge_equals_unsplit, pin_merge_identities]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_thread_count_does_not_change_result(oracle_lib):
    p = wl.make_problem("threads", [33, 70, 5, 128], Hq=8, Hkv=2, D=32, page_size=16,
                        num_pages=24, seed=18)
    a = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, nthreads=1)
    b = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_oracle_rejects_bad_problems(oracle_lib):
    p = wl.tiny()
    bad = p.block_table.copy()
    bad[0, 0] = p.num_pages  # page id out of range
    with pytest.raises(ValueError):
        oracle.decode(p.q, p.k_pages, p.v_pages, bad, p.seq_lens)
    with pytest.raises(ValueError):  # longer than the table allows
        oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, np.array([37, 7 * 16 + 1], np.int32))


# --- planted mistakes ------------------------------------------------------------------

MUTANTS = {
    "scale_dropped": ("const double scale = 1.0 / sqrt((double)D);", "const double scale = 1.0;"),
    "head_map_modulo": ("const int kvh = h / G;", "const int kvh = h % p->Hkv;"),
    "lse_base_two": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "slots_reversed": ("int slot = t % p->page_size;", "int slot = p->page_size - 1 - t % p->page_size;"),
    "no_normalisation": ("for (int d = 0; d < D; ++d) out[d] /= l;", ""),
    "merge_unweighted": ("double w = exp(lse_parts[s] - M);", "double w = 1.0;"),
    "off_by_one_last_token": ("for (int t = t_begin; t < t_end; ++t) {\n        double w",
                              "for (int t = t_begin; t < t_end - (t_end - t_begin > 1); ++t) {\n        double w"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    """A mistake planted in a copy of the oracle must fail at least one pin."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / f"mutant_{name}.c"
    mutant_src.write_text(src.replace(old, new))
    path = oracle.build(force=True, src=str(mutant_src), out=str(tmp_path / f"libmutant_{name}.so"))
    lib = oracle.load(path)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
