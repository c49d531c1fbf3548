"""Seeded synthetic inputs for paged decode attention.

This module only draws numbers: sequence lengths, page placement and bf16
tensors.  It holds none of the attention arithmetic, so both the CUDA path and
the CPU oracle may take their inputs from it.

Workload shapes follow the traces that "PersistentKV: Page-Aware Decode
Scheduling for Long-Context LLM Serving on Commodity GPUs" (gist.science
summary, Methodology section 3 "Evaluation Protocol") describes: batch-1 long
context, small mixed-length batches, and a high active batch; plus the
many-sessions continuous workload of "WPK persistent kernel" (dotwave.ai,
Figure 01).  Those traces are not published, so these seeded recipes stand in
for them.

Recipe (every workload):
  1. rng = numpy.random.default_rng(seed); seed 20260623 is the held-out seed
     and 20260622 the calibration seed of the PersistentKV summary (Results).
  2. Sequence lengths are drawn first (when random), then the pool size is
     fixed, then rng.permutation(num_pages) places pages: row 0 takes the first
     P_0 entries of the permutation, row 1 the next P_1, and so on, so block
     tables are non-contiguous and shuffled.  Unused table entries are -1.
  3. q [B][Hq][D], then K pages, then V pages [NP][ps][Hkv][D] are drawn
     float32 standard normal and rounded to the nearest bf16 (ties to even).
     Every page of the pool is filled, used or not.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HELD_OUT_SEED = 20260623
CALIBRATION_SEED = 20260622


@dataclasses.dataclass
class Problem:
    name: str
    q: np.ndarray            # uint16 bf16 bits [B][Hq][D]
    k_pages: np.ndarray      # uint16 [NP][ps][Hkv][D]
    v_pages: np.ndarray      # uint16 [NP][ps][Hkv][D]
    block_table: np.ndarray  # int32 [B][max_pages], -1 where unused
    seq_lens: np.ndarray     # int32 [B]
    page_size: int
    num_splits: int = 0      # requested split count (0 = planner's choice)
    free_pages: np.ndarray | None = None  # pool pages not in any table (continuous workload)
    notes: str = ""

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def Hq(self) -> int:
        return self.q.shape[1]

    @property
    def D(self) -> int:
        return self.q.shape[2]

    @property
    def Hkv(self) -> int:
        return self.k_pages.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_pages.shape[0]

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]

    def kv_bytes(self) -> int:
        """K and V bytes the step must read: sum_b N_b * Hkv * D * 2 (K, V) * 2 B."""
        return int(np.sum(self.seq_lens, dtype=np.int64)) * self.Hkv * self.D * 2 * 2


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_to_float32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    return round_to_bf16(rng.standard_normal(size=shape, dtype=np.float32))


def _place_pages(rng, seq_lens, page_size, num_pages, max_pages):
    """Assign each row's pages from one seeded permutation of the pool."""
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((len(seq_lens), max_pages), -1, dtype=np.int32)
    cursor = 0
    for b, n in enumerate(seq_lens):
        p = -(-int(n) // page_size)
        table[b, :p] = perm[cursor:cursor + p]
        cursor += p
    if cursor > num_pages:
        raise ValueError("pool too small")
    return table, perm[cursor:]


def make_problem(name: str, seq_lens, *, Hq: int, Hkv: int, D: int, page_size: int,
                 num_pages: int, max_pages: int | None = None, seed: int = HELD_OUT_SEED,
                 rng: np.random.Generator | None = None, num_splits: int = 0,
                 notes: str = "") -> Problem:
    rng = rng if rng is not None else np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    if max_pages is None:
        max_pages = max(1, max((-(-int(n) // page_size) for n in seq_lens), default=1))
    table, free = _place_pages(rng, seq_lens, page_size, num_pages, max_pages)
    B = len(seq_lens)
    q = bf16_normal(rng, (B, Hq, D))
    k = bf16_normal(rng, (num_pages, page_size, Hkv, D))
    v = bf16_normal(rng, (num_pages, page_size, Hkv, D))
    return Problem(name, q, k, v, table, seq_lens, page_size, num_splits, free, notes)


# --- the five workloads --------------------------------------------------------------

def tiny(seed: int = HELD_OUT_SEED) -> Problem:
    """Batch 2, lengths 37 and 100, 4 query heads / 1 KV head, D 64, ps 16, 16-page pool."""
    return make_problem("tiny", [37, 100], Hq=4, Hkv=1, D=64, page_size=16, num_pages=16,
                        seed=seed, notes="split counts 1, 2, 4 are all checked")


def batch1_long(seed: int = HELD_OUT_SEED) -> Problem:
    """1 x 32768 tokens, 32/8 heads, D 128, ps 16, 2048 pages drawn from a 4096-page pool, S 32."""
    return make_problem("batch1_long_32k", [32768], Hq=32, Hkv=8, D=128, page_size=16,
                        num_pages=4096, seed=seed, num_splits=32)


def mixed_lengths(seed: int = HELD_OUT_SEED):
    """(lengths, rng): the rng continues into page placement and tensors."""
    rng = np.random.default_rng(seed)
    return np.floor(np.exp(rng.uniform(math.log(512), math.log(32768), size=8))).astype(np.int32), rng


def mixed(seed: int = HELD_OUT_SEED) -> Problem:
    """8 rows, lengths floor(exp(U(ln 512, ln 32768))), 32/8 heads, D 128, pool = 1.25 x pages."""
    lens, rng = mixed_lengths(seed)
    pages = int(sum(-(-int(n) // 16) for n in lens))
    return make_problem("mixed_b8", lens, Hq=32, Hkv=8, D=128, page_size=16,
                        num_pages=int(math.ceil(pages * 1.25)), rng=rng)


def high_batch(seed: int = HELD_OUT_SEED) -> Problem:
    """64 x 4096 tokens, 32/8 heads, D 128, shuffled tables, pool exactly the used pages."""
    return make_problem("high_batch_64x4096", [4096] * 64, Hq=32, Hkv=8, D=128, page_size=16,
                        num_pages=64 * 256, seed=seed)


def continuous(seed: int = HELD_OUT_SEED, steps: int = 200, sessions: int = 56) -> Problem:
    """56 sessions, lengths U[1024, 8192], room for `steps` appended tokens each;
    pool = 1.25 x sum_b ceil((N_b + steps) / 16); new pages come from `free_pages`."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1024, 8192, size=sessions, endpoint=True).astype(np.int32)
    need = int(sum(-(-(int(n) + steps) // 16) for n in lens))
    max_pages = max(-(-(int(n) + steps) // 16) for n in lens)
    return make_problem("continuous_56", lens, Hq=32, Hkv=8, D=128, page_size=16,
                        num_pages=int(math.ceil(need * 1.25)), max_pages=max_pages, rng=rng,
                        notes=f"{steps} steps of append + decode")


# --- the trace families of the PersistentKV summary (Methodology section 3) ---------------
#
# The summary names Bucketed, Bimodal, Uniform and Zipf-like traces "designed to isolate
# context length, active batch size, and length raggedness" but publishes none of their
# parameters.  These are the readings taken here (lengths in tokens, at most 32768):
#   uniform   N ~ U[512, 32768]
#   bimodal   each row short, N ~ U[256, 2048], or long, N ~ U[16384, 32768], with p = 1/2
#   zipf      N = 512 * k with k Zipf(1.3) distributed, truncated to k <= 64
#   bucketed  N drawn from the buckets {1024, 4096, 16384, 32768}
TRACE_KINDS = ("uniform", "bimodal", "zipf", "bucketed")


def trace_lengths(kind: str, batch: int, rng: np.random.Generator) -> np.ndarray:
    if kind == "uniform":
        n = rng.integers(512, 32768, size=batch, endpoint=True)
    elif kind == "bimodal":
        long_rows = rng.random(batch) < 0.5
        n = np.where(long_rows, rng.integers(16384, 32768, size=batch, endpoint=True),
                     rng.integers(256, 2048, size=batch, endpoint=True))
    elif kind == "zipf":
        k = rng.zipf(1.3, size=batch)
        n = 512 * np.minimum(k, 64)
    elif kind == "bucketed":
        n = rng.choice(np.array([1024, 4096, 16384, 32768]), size=batch)
    else:
        raise ValueError(kind)
    return np.asarray(n, dtype=np.int32)


def trace(kind: str, batch: int, seed: int = HELD_OUT_SEED) -> Problem:
    """A trace-family batch: 32/8 heads, D 128, 16-token pages, pool 1.25 x the pages in use."""
    rng = np.random.default_rng(seed)
    lens = trace_lengths(kind, batch, rng)
    pages = int(sum(-(-int(n) // 16) for n in lens))
    return make_problem(f"{kind}_b{batch}", lens, Hq=32, Hkv=8, D=128, page_size=16,
                        num_pages=int(math.ceil(pages * 1.25)), rng=rng)


WORKLOADS = {
    "tiny": tiny,
    "batch1_long": batch1_long,
    "mixed": mixed,
    "high_batch": high_batch,
    "continuous": continuous,
}


def new_tokens(rng: np.random.Generator, B: int, Hkv: int, D: int):
    """One step's appended K and V tokens, bf16 bits [B][Hkv][D] each."""
    return bf16_normal(rng, (B, Hkv, D)), bf16_normal(rng, (B, Hkv, D))
