"""GPU: the allocation-free decode entry point.

pgqa_decode_static_scratch is for callers that cannot allocate device memory
(for example code running while a CUDA graph is captured, or runtimes that own
all device memory through their own allocator).  It keeps its work list and
split partials in a fixed array inside the library.  This test calls it through
the C ABI twice in a row and checks both results against the plan/run entry
point on the same inputs, with the tolerances the other parity tests use.
It lives in its own file, collected last, so that a failure here never stops
the rest of the suite.
"""
import numpy as np
import pytest
import torch

import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

CASES = [
    # lengths, page size, Hq, Hkv, head_dim, dtype, pool pages, splits
    ([0, 1, 17, 300, 1000, 64], 16, 14, 2, 64, "bf16", 256, 3),
    ([5, 257, 2048, 4099], 256, 12, 2, 128, "fp16", 64, 8),
    ([301] * 32, 16, 14, 2, 64, "bf16", 1024, 1),
]


def plan_run(w, dev):
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                   max_batch=w.batch, max_q_rows=w.rows)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages)
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    out = plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out_dtype=torch.float32, lse=lse)
    torch.cuda.synchronize()
    plan.close()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_plan_run_twice(case):
    lens, ps, hq, hkv, d, dtype, pages, splits = CASES[case]
    w = W.custom("noalloc", lens, ps, hq, hkv, d, dtype, pages, seed=40 + case)
    dev = H.to_device(w)
    ref_out, ref_lse = plan_run(w, dev)
    indptr = torch.from_numpy(w.kv_indptr).cuda()
    last = torch.from_numpy(w.last_page_len).cuda()
    outs = []
    for _ in range(2):  # the second call reuses the array the first one left behind
        out = torch.full(dev["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full(dev["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pg.decode_static_scratch(dev["q"], dev["k_pool"], dev["v_pool"], indptr, dev["kv_indices"], last,
                                 splits, out=out, lse=lse)
        torch.cuda.synchronize()
        o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
        H.compare(o, l, ref_out, ref_lse, f"static scratch case {case}")
        outs.append((o, l))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert pg.read_device_flags() == 0


def test_static_scratch_rejects_oversized_request():
    w = W.custom("big", [16] * 8, 16, 8, 1, 128, "bf16", 16, seed=1)
    dev = H.to_device(w)
    indptr = torch.from_numpy(w.kv_indptr).cuda()
    last = torch.from_numpy(w.last_page_len).cuda()
    q = torch.zeros(4096, 8, 128, dtype=torch.bfloat16, device="cuda")
    big_indptr = torch.zeros(4097, dtype=torch.int32, device="cuda")
    big_last = torch.zeros(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(pg.PagedGQAError) as e:
        pg.decode_static_scratch(q, dev["k_pool"], dev["v_pool"], big_indptr, dev["kv_indices"], big_last, 256,
                                 out_dtype=torch.float32)
    assert e.value.name == "PGQA_ERR_CAPACITY"
    del indptr, last
