"""pkv: single-token GQA decode attention over a block-table paged KV cache,
hand-written CUDA for GB300 (sm_103a) behind a small C ABI (include/pkv.h).

The CUDA library is loaded on first use by ``paged_kv_decode_block_gb300.pkv``;
importing this package alone touches no GPU code, so the seeded input
generators in ``workloads`` can be used on any machine.
"""
__all__ = ["workloads", "pkv"]
