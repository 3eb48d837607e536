"""GPU: pgqa_append_run (append of the step's new rows + attention in one launch)
against the CPU oracle's append followed by its attention."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def fused_gpu(w, pool_stable=False, out_dtype=torch.float32, **plan_opts):
    dev = H.to_device(w)
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                   max_batch=w.batch, max_q_rows=w.rows, **plan_opts)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                causal=w.causal, kv_indices_host=w.kv_indices)
    out = torch.empty(dev["q"].shape, dtype=out_dtype, device="cuda")
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    plan.append_run(dev["k_new"], dev["v_new"], dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse,
                    pool_stable=pool_stable)
    torch.cuda.synchronize()
    info = plan.info()
    plan.close()
    assert pg.read_device_flags() == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), dev, info


def check_pool(w, dev):
    kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
    oracle.get().kv_append(kp, vp, W.raw16(w.k_new), W.raw16(w.v_new), w.slot_mapping)
    assert np.array_equal(W.raw16(dev["k_pool"]), kp), "fused append K rows differ"
    assert np.array_equal(W.raw16(dev["v_pool"]), vp), "fused append V rows differ"


@pytest.mark.parametrize("opts", [{}, {"split_tokens": 64}, {"max_splits": 1}, {"pipeline_stages": 1},
                                  {"pipeline_stages": 2}])
@pytest.mark.parametrize("pool_stable", [False, True])
def test_fused_decode_step(opts, pool_stable):
    w = W.qwen05_decode(batch=32, cached=300, num_pages=1024)
    ro, rl = H.oracle_outputs(w)
    out, lse, dev, info = fused_gpu(w, pool_stable=pool_stable, **opts)
    H.compare(out, lse, ro, rl, f"fused decode {opts} stable={pool_stable}")
    check_pool(w, dev)


@pytest.mark.parametrize("head_dim,page_size,dtype,heads", [(128, 256, "fp16", 12), (64, 64, "bf16", 12),
                                                             (128, 16, "bf16", 12), (64, 16, "bf16", 32),
                                                             (128, 32, "fp16", 22)])
def test_fused_shapes(head_dim, page_size, dtype, heads):
    w = W.custom("fz", [1, 2, 17, 33, 200, 700], page_size, heads, 2, head_dim, dtype, 64,
                 seed=head_dim + page_size + heads)
    H.new_rows_for_query_rows(w)
    ro, rl = H.oracle_outputs(w)
    out, lse, dev, _ = fused_gpu(w, split_tokens=64)
    H.compare(out, lse, ro, rl, f"fused d{head_dim} ps{page_size} {dtype} Hq{heads}")
    check_pool(w, dev)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("prefill_kernel", ["tcgen05", "mma_sync"])
def test_fused_multi_row(causal, prefill_kernel):
    """A chunk of L query rows per request appends L rows (the ragged step)."""
    w = W.custom("fzr", [40, 7, 300, 64], 16, 14, 2, 64, "bf16", 64, seed=11, qo_lens=[13, 1, 5, 64],
                 causal=causal)
    H.new_rows_for_query_rows(w)
    ro, rl = H.oracle_outputs(w)
    out, lse, dev, _ = fused_gpu(w, split_tokens=64, prefill_kernel=prefill_kernel)
    H.compare(out, lse, ro, rl, f"fused multi-row causal={causal} {prefill_kernel}")
    check_pool(w, dev)


def test_fused_native_out_dtype():
    w = W.qwen05_decode(batch=8, cached=100, num_pages=128)
    ro, rl = H.oracle_outputs(w)
    out, lse, _, _ = fused_gpu(w, out_dtype=torch.bfloat16)
    H.compare(out, lse, ro, rl, "fused bf16 out", out_dtype="bf16")


def test_fused_rejects_cuda_core_plan_and_short_requests():
    w = W.qwen05_decode(batch=4, cached=10, num_pages=16)
    dev = H.to_device(w)
    plan = pg.Plan(14, 2, 64, 16, torch.bfloat16, 4, 4, decode_kernel="cuda_core")
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages)
    with pytest.raises(pg.PagedGQAError) as e:
        plan.append_run(dev["k_new"], dev["v_new"], dev["q"], dev["k_pool"], dev["v_pool"])
    assert e.value.name == "PGQA_ERR_UNSUPPORTED"
    # 3 query rows on a request with 2 keys: nowhere to put the third new row
    w2 = W.custom("short", [2], 16, 4, 2, 64, "bf16", 4, seed=1, qo_lens=[3], causal=True)
    d2 = H.to_device(w2)
    p2 = pg.Plan(4, 2, 64, 16, torch.bfloat16, 1, 3)
    p2.update(w2.kv_indptr, w2.last_page_len, d2["kv_indices"], w2.num_pages, qo_indptr=w2.qo_indptr,
              causal=True)
    kn = torch.zeros(3, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pg.PagedGQAError) as e:
        p2.append_run(kn, kn, d2["q"], d2["k_pool"], d2["v_pool"])
    assert e.value.name == "PGQA_ERR_INVALID_ARG"


@pytest.mark.parametrize("head_dim", [64, 128])
def test_wide_form_boundaries(head_dim):
    """Rows around the decode kernel's wide form (ten warps of one tile: up to 320 keys at
    d 64, 160 at d 128), whose appended row lands in every warp's tile in turn: the fused
    step and append-then-run against the oracle, under the plan's choice, the wide form
    forced and forced splits."""
    tile = 32 if head_dim == 64 else 16
    lens = sorted({n for k in range(1, 11) for n in (k * tile - 1, k * tile, k * tile + 1)})
    w = W.custom("wideb", lens, 16, 14, 2, head_dim, "bf16", 512, seed=head_dim + 11, append_last=True)
    ro, rl = H.oracle_outputs(w)
    for opts in ({}, {"pipeline_stages": 1}, {"split_tokens": 2 * tile}):
        out, lse, dev, _ = fused_gpu(w, **opts)
        H.compare(out, lse, ro, rl, f"fused wide boundaries d{head_dim} {opts}")
        check_pool(w, dev)
        out, lse, _ = H.gpu_outputs(w, **opts)
        H.compare(out, lse, ro, rl, f"wide boundaries d{head_dim} {opts}")
