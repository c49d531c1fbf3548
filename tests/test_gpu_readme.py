"""The Python example of README.md, run as written (seeded), and checked against
the fp64 oracle within 2e-3 / 1e-4."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_block_gb300 import pkv
from pkv_testutil import assert_close

pytestmark = pytest.mark.gpu


def test_readme_example():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.manual_seed(0)
    # --- the README example
    B, Hq, Hkv, D, ps, max_pages, num_pages = 2, 32, 8, 128, 16, 64, 128
    k = torch.randn(num_pages, ps, Hkv, D, device="cuda").bfloat16()
    v = torch.randn_like(k)
    q = torch.randn(B, Hq, D, device="cuda").bfloat16()
    lens_h = [1000, 37]
    table_h = torch.full((B, max_pages), -1, dtype=torch.int32)
    table_h[0, :63] = torch.arange(63)
    table_h[1, :3] = torch.arange(63, 66)
    table, lens = table_h.cuda(), torch.tensor(lens_h, dtype=torch.int32, device="cuda")
    out = torch.empty(B, Hq, D, device="cuda")
    lse = torch.empty(B, Hq, device="cuda")

    plan = pkv.Plan(lens_h, table_h.numpy(), ps, B=B, Hq=Hq, Hkv=Hkv, D=D,
                    max_pages=max_pages, num_pages=num_pages)
    pkv.decode(q, k, v, table, lens, plan, out, lse)
    # ---
    torch.cuda.synchronize()
    assert plan.status() == 0
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    ref_out, ref_lse = oracle.decode(bits(q), bits(k), bits(v), table_h.numpy(), np.array(lens_h, np.int32),
                                     nthreads=8)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, what="README example")
    plan.close()
