"""GPU: back-to-back calls on one plan, whose split partials share the plan's
buffers.

Every call's slices store into the same partial slots, and the merge of one call
overlaps the start of the next call's kernels (programmatic dependent launch: a
kernel's prologue and, with POOL_STABLE, its K/V loads run before the previous
grid ends; its stores only after).  These tests run one plan several times with
a different q each time and no synchronisation between the calls, so a slice
that overwrote partials an earlier merge was still reading, or a merge that read
before its partials were stored, shows up as a wrong output.  Both merge launch
shapes (one warp per head for at most 32 slices, a block per 32 channels beyond)
and split prefill rows are covered.
"""
import pytest
import torch

import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

CASES = {
    # decode rows, at most 32 slices each: the warp-per-head merge
    "warp_merge": (dict(kv_lens=[2000, 37, 1500, 5, 640, 1], page_size=16, num_qo_heads=12, num_kv_heads=2,
                        head_dim=128, dtype="fp16", num_pages=512, seed=3), {"split_tokens": 64}),
    # 125 slices on the longest row: the block-per-channel-chunk merge
    "block_merge": (dict(kv_lens=[2000, 300, 17], page_size=16, num_qo_heads=14, num_kv_heads=2,
                         head_dim=64, dtype="bf16", num_pages=256, seed=4), {"split_tokens": 16}),
    # a causal chunk cut into key slices next to split decode rows
    "ragged": (dict(kv_lens=[700, 1200, 90, 1100], page_size=16, num_qo_heads=14, num_kv_heads=2,
                    head_dim=64, dtype="bf16", num_pages=512, seed=5, qo_lens=[1, 200, 1, 1], causal=True),
               {"split_tokens": 128, "prefill_splits": 4}),
}


def fresh_q(w, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(w.q.shape, generator=gen).to(w.q.dtype)


@pytest.mark.parametrize("pool_stable", [False, True])
@pytest.mark.parametrize("case", sorted(CASES))
def test_back_to_back_calls_on_one_plan(case, pool_stable):
    spec, opts = CASES[case]
    w = W.custom(case, **spec)
    dev = H.to_device(w)
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                   max_batch=w.batch, max_q_rows=w.rows, **opts)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                causal=w.causal, kv_indices_host=w.kv_indices)
    info = plan.info()
    assert info["num_merge_tasks"] > 0
    qs = [fresh_q(w, 100 + k) for k in range(3)]
    outs, lses = [], []
    pg.read_device_flags(clear=True)
    for q in qs:  # no synchronisation between the calls
        qd = q.cuda()
        out = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
        lse = torch.empty(qd.shape[:2], dtype=torch.float32, device="cuda")
        plan.run(qd, dev["k_pool"], dev["v_pool"], out=out, lse=lse, pool_stable=pool_stable)
        outs.append(out)
        lses.append(lse)
    # and once more into the first buffers
    plan.run(qs[0].cuda(), dev["k_pool"], dev["v_pool"], out=outs[0], lse=lses[0], pool_stable=pool_stable)
    torch.cuda.synchronize()
    plan.close()
    assert pg.read_device_flags() == 0
    for k, q in enumerate(qs):
        w.q = q
        ro, rl = H.oracle_outputs(w)
        H.compare(outs[k].double().cpu().numpy(), lses[k].double().cpu().numpy(), ro, rl, f"{case} call {k}")
