"""fp64 CPU oracle for paged GQA decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only importers.  Nothing here is shared
with the CUDA path, and the product library never imports this package.

Contents
--------
``decode``      full attention per (row, query head), C in fp64 (pkv_oracle.c)
``partial``     the partial softmax state of one split, C in fp64
``merge``       exact log-sum-exp merge of partial states, C in fp64
``enumerate_queue`` / ``enumerate_padded_grid`` / ``enumerate_direct``   work-tile lists (queue.py)
``append``      the KV-cache append of one token per (row, KV head) (append.py)

Everything follows "PersistentKV: Page-Aware Decode Scheduling for Long-Context
LLM Serving on Commodity GPUs" (gist.science summary), Technical Summary,
Methodology section 1; the readings taken where that page is silent are listed
in the header of each file.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
things other than itself (a library attention routine, closed forms, worked
examples in ``tests/golden/``, invariants and brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

from .queue import enumerate_queue, enumerate_padded_grid, enumerate_direct, chunk_pages_for_splits  # noqa: F401
from .append import append  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle with gcc into a shared library; returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *extra_flags, src, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
    i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
    f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
    ci = ctypes.c_int
    lib.pkv_oracle_decode.restype = ci
    lib.pkv_oracle_decode.argtypes = [u16p, u16p, u16p, i32p, i32p] + [ci] * 7 + [f64p, f64p, ci]
    lib.pkv_oracle_partial.restype = ci
    lib.pkv_oracle_partial.argtypes = [u16p, u16p, u16p, i32p, i32p] + [ci] * 7 + [ci] * 4 + [f64p, f64p]
    lib.pkv_oracle_merge.restype = None
    lib.pkv_oracle_merge.argtypes = [f64p, f64p, ci, ci, f64p, f64p]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  A path loads another build of it."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _geometry(q, k_pages, block_table, seq_lens):
    B, Hq, D = q.shape
    NP, ps, Hkv, D2 = k_pages.shape
    if D2 != D:
        raise ValueError("head_dim of q and pages differ")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("batch size of block_table/seq_lens differs from q")
    return B, Hq, Hkv, D, ps, block_table.shape[1], NP


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def decode(q, k_pages, v_pages, block_table, seq_lens, nthreads: int = 1, lib=None):
    """Full paged decode attention.  q: uint16 bf16 bits [B][Hq][D];
    k_pages/v_pages: uint16 [NP][ps][Hkv][D]; block_table int32 [B][max_pages];
    seq_lens int32 [B].  Returns (out float64 [B][Hq][D], lse float64 [B][Hq])."""
    lib = lib or load()
    q, k_pages, v_pages = _c(q, np.uint16), _c(k_pages, np.uint16), _c(v_pages, np.uint16)
    block_table, seq_lens = _c(block_table, np.int32), _c(seq_lens, np.int32)
    B, Hq, Hkv, D, ps, max_pages, NP = _geometry(q, k_pages, block_table, seq_lens)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.pkv_oracle_decode(q, k_pages, v_pages, block_table, seq_lens, B, Hq, Hkv, D, ps,
                               max_pages, NP, out, lse, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return out, lse


def partial(q, k_pages, v_pages, block_table, seq_lens, b, kvh, token_begin, token_end, lib=None):
    """Partial state of tokens [token_begin, min(token_end, N_b)) of row b for the
    G query heads of KV head kvh.  Returns (o float64 [G][D], lse float64 [G])."""
    lib = lib or load()
    q, k_pages, v_pages = _c(q, np.uint16), _c(k_pages, np.uint16), _c(v_pages, np.uint16)
    block_table, seq_lens = _c(block_table, np.int32), _c(seq_lens, np.int32)
    B, Hq, Hkv, D, ps, max_pages, NP = _geometry(q, k_pages, block_table, seq_lens)
    G = Hq // Hkv
    o = np.zeros((G, D), np.float64)
    lse = np.zeros((G,), np.float64)
    rc = lib.pkv_oracle_partial(q, k_pages, v_pages, block_table, seq_lens, B, Hq, Hkv, D, ps,
                                max_pages, NP, int(b), int(kvh), int(token_begin), int(token_end),
                                o, lse)
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return o, lse


def merge(o_parts, lse_parts, lib=None):
    """Exact LSE merge of S partial states of one head: o_parts [S][D], lse_parts [S]."""
    lib = lib or load()
    o_parts = _c(o_parts, np.float64)
    lse_parts = _c(lse_parts, np.float64)
    S, D = o_parts.shape
    out = np.zeros((D,), np.float64)
    lse = np.zeros((1,), np.float64)
    lib.pkv_oracle_merge(o_parts, lse_parts, S, D, out, lse)
    return out, float(lse[0])


def available_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


if __name__ == "__main__":  # build entry point: python -m oracle
    print(build(force="--force" in sys.argv))
