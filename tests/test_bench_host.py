"""Host-side pieces of bench.py that its GPU run depends on, checked on CPU:
the route label of the roofline line, the workload part of the config, the
single-threaded oracle step's time gate and the parity gate."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from paged_kv_decode_block_gb300 import pkv  # noqa: E402
from paged_kv_decode_block_gb300 import workloads as wl  # noqa: E402

SMALL = dict(Hq=32, Hkv=8, D=128)


def _info(lens, **opts):
    lens = np.asarray(lens, np.int32)
    max_pages = max(1, int(-(-lens.max() // 16)))
    return pkv.dry_run(lens, None, 16, B=len(lens), **SMALL, max_pages=max_pages,
                       num_pages=int(sum(-(-int(n) // 16) for n in lens)) + 1, num_sms=152, ctas_per_sm=2,
                       **opts)[0]


@pytest.mark.parametrize("lens,opts,words", [
    ([32768], dict(force_mode="split_queue", num_splits=32),
     "split partials over the compact queue, LSE merge fused"),
    (wl.mixed_lengths()[0], dict(force_mode="split_padded"),
     "split partials over the padded split grid, LSE merge fused"),
    ([4096] * 64, dict(), "one tile per (row, KV head), finalised in place"),
    ([32768], dict(force_mode="split_queue", num_splits=32, separate_merge=True),
     "split partials over the compact queue, LSE merge in its own launch"),
    ([300, 40], dict(force_mode="split_queue", num_splits=1), "split partials over the compact queue"),
    ([1024, 8192], dict(force_mode="persistent", num_splits=1),
     "persistent CTAs draining the queue"),
])
def test_route_words_name_the_launch(lens, opts, words):
    assert bench.route_words(_info(lens, **opts)) == words


def test_workload_config_of_the_tiny_case():
    p, opts = bench.build_workload("tiny")
    cfg = bench.workload_config(p, "tiny", world=2)
    assert cfg["batch"] == 2 and cfg["q_heads"] == 4 and cfg["kv_heads"] == 1 and cfg["head_dim"] == 64
    assert cfg["seq_lens"] == "sum 137" and cfg["page_size"] == 16
    assert cfg["parallelism"].startswith("replicas x2")
    assert opts == dict(force_mode="split_queue", num_splits=4)


def test_single_thread_step_is_gated_by_its_estimate():
    p = wl.tiny()
    assert bench.single_thread_oracle(p, p.kv_bytes(), estimate_s=16.0) is None
    got = bench.single_thread_oracle(p, p.kv_bytes(), estimate_s=0.01)
    assert got["cores"] == 1 and got["unit"] == "GB/s" and got["value"] > 0


def test_parity_gate_passes_the_oracle_and_catches_an_error():
    p = wl.tiny()
    out, lse = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens)
    out, lse = out.astype(np.float32), lse.astype(np.float32)
    assert bench.parity_gate(p, out, lse, 1)[0]
    bad = out.copy()
    bad[1, 2, 3] += 3e-3
    assert not bench.parity_gate(p, bad, lse, 1)[0]


def test_trace_workload_names():
    assert bench.parse_trace_name("batch1_long") is None
    assert bench.parse_trace_name("trace:zipf:8") == ("zipf", 8)
    for bad in ("trace:zipf", "trace:normal:4", "trace:uniform:0", "trace:uniform:x"):
        with pytest.raises(ValueError):
            bench.parse_trace_name(bad)
    p, opts = bench.build_workload("trace:bimodal:4")
    ref = wl.trace("bimodal", 4)
    assert opts == {} and p.name == "bimodal_b4" and np.array_equal(p.seq_lens, ref.seq_lens)


def test_product_package_never_imports_the_oracle():
    """Only the tests, the smoke entry and bench.py may import oracle/."""
    pkg = os.path.join(ROOT, "paged_kv_decode_block_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cpp", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "pkv_oracle" not in text, f


def test_phase_summary_of_synthetic_rows():
    """Two CTAs: one streams and merges, one streams and only arrives."""
    rows = np.zeros((2, pkv.TRACE_WORDS), np.uint64)
    base = 10_000_000
    # tiles, sm, entry, wait, first, stream_end, combine, arrived, merge_end, exit
    rows[0, :10] = [1, 3, base - 500, base, base + 1500, base + 20500, base + 21000, base + 22000, base + 24000,
                    base + 24100]
    rows[1, :10] = [1, 4, base - 400, base + 100, base + 1700, base + 20300, base + 20700, base + 21500, 0,
                    base + 21600]
    s = bench.phase_summary(rows, pkv)
    assert s["ctas"] == 2 and s["ctas_with_tiles"] == 2
    assert s["wait_to_first_block"] == 1.55 and s["stream"] == 18.8 and s["combine"] == 0.45
    assert s["arrival"] == 0.9 and s["merge"] == 2.0 and s["launch_span"] == 24.1 and s["last_merge_end"] == 24.0
    assert s["wait_released_spread"] == 0.1 and s["stream_end_median_to_last"] == 0.1
