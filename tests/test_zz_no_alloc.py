"""GPU: the allocation-free decode entry point.

pgqa_decode_static_scratch serves callers of this library that cannot allocate
device memory: processes whose device memory is reserved up front and handed
out by another allocator, and embedded or real-time hosts that forbid
allocation after start-up.  It keeps its work list and split partials in a
fixed array inside the library.  These tests call it through the C ABI twice
in a row (the second call finds the array as the first left it) and check both
results element by element against the CPU oracle with the tolerances the
other parity tests use, and against the plan/run entry point on the same
inputs.  Malformed device page tables must be caught before any read through
them: the bad requests get no keys and the device flag is raised.
The file is collected last, so that a failure here never stops the rest of the
suite.
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
    ([0, 0, 0], 16, 14, 2, 64, "bf16", 8, 2),  # every request empty: kv_indices has no entries
]

FLAG_PAGE_INDEX = 1


def plan_run(w, dev):
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                   max_batch=w.batch, max_q_rows=w.rows)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages)
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    out = plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out_dtype=torch.float32, lse=lse)
    torch.cuda.synchronize()
    plan.close()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def static_call(dev, indptr, indices, last, splits):
    out = torch.full(dev["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full(dev["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pg.decode_static_scratch(dev["q"], dev["k_pool"], dev["v_pool"], indptr, indices, last, splits,
                             out=out, lse=lse)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_oracle_and_plan_run_twice(case):
    lens, ps, hq, hkv, d, dtype, pages, splits = CASES[case]
    w = W.custom("noalloc", lens, ps, hq, hkv, d, dtype, pages, seed=40 + case)
    pg.read_device_flags(clear=True)
    dev = H.to_device(w)
    ro, rl = H.oracle_outputs(w)
    po, pl = plan_run(w, dev)
    indptr = torch.from_numpy(w.kv_indptr).cuda()
    last = torch.from_numpy(w.last_page_len).cuda()
    outs = []
    for call in range(2):  # the second call reuses the array the first one left behind
        o, l = static_call(dev, indptr, dev["kv_indices"], last, splits)
        H.compare(o, l, ro, rl, f"static scratch case {case} call {call} vs oracle")
        H.compare(o, l, po, pl, f"static scratch case {case} call {call} vs plan/run")
        outs.append((o, l))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert pg.read_device_flags() == 0


def _expected_with_empty(ro, rl, bad_rows):
    eo, el = ro.copy(), rl.copy()
    eo[bad_rows] = 0.0
    el[bad_rows] = -np.inf
    return eo, el


# request lengths [0, 17, 300, 5] at page 16 -> pages [0, 2, 19, 1], kv_indptr [0, 0, 2, 21, 22]
MALFORMED = {
    # name: (kv_indptr, last_page_len edits, entries of kv_indices passed, requests that get no keys)
    "decreasing": ([0, 0, 2, 21, 20], {}, 22, [3]),
    "negative": ([0, -5, 2, 21, 22], {}, 22, [0, 1]),
    "past_end": ([0, 0, 2, 21, 22], {}, 21, [3]),
    "empty_with_last": ([0, 0, 2, 21, 22], {0: 3}, 22, [0]),
}


@pytest.mark.parametrize("name", sorted(MALFORMED))
def test_static_scratch_malformed_table_is_caught_before_use(name):
    """Each table is wrong in one place; the requests it touches come back empty
    (out 0, lse -inf) with PGQA_FLAG_PAGE_INDEX raised, and the others are right."""
    w = W.custom("noalloc-bad", [0, 17, 300, 5], 16, 14, 2, 64, "bf16", 64, seed=9)
    assert list(w.kv_indptr) == [0, 0, 2, 21, 22]
    indptr_l, last_edits, n_idx, bad = MALFORMED[name]
    pg.read_device_flags(clear=True)
    dev = H.to_device(w)
    ro, rl = H.oracle_outputs(w)
    eo, el = _expected_with_empty(ro, rl, bad)
    last = w.last_page_len.copy()
    for b, v in last_edits.items():
        last[b] = v
    o, l = static_call(dev, torch.tensor(indptr_l, dtype=torch.int32, device="cuda"),
                       dev["kv_indices"][:n_idx].contiguous(), torch.from_numpy(last).cuda(), 2)
    H.compare(o, l, eo, el, f"malformed table '{name}'")
    assert pg.read_device_flags() & FLAG_PAGE_INDEX


def test_static_scratch_rejects_oversized_request():
    w = W.custom("big", [16] * 8, 16, 8, 1, 128, "bf16", 16, seed=1)
    dev = H.to_device(w)
    q = torch.zeros(4096, 8, 128, dtype=torch.bfloat16, device="cuda")
    big_indptr = torch.zeros(4097, dtype=torch.int32, device="cuda")
    big_last = torch.zeros(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(pg.PagedGQAError) as e:
        pg.decode_static_scratch(q, dev["k_pool"], dev["v_pool"], big_indptr, dev["kv_indices"], big_last, 256,
                                 out_dtype=torch.float32)
    assert e.value.name == "PGQA_ERR_CAPACITY"
