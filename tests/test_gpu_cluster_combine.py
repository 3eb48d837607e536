"""GPU: split decode rows combined inside thread-block clusters (split_combine = a
cluster size) against the CPU oracle.

Every split row's slices run as consecutive CTAs of one cluster; the row's last
slice reads the others' (O, log-sum-exp) from their shared memory and writes the
row, with no merge grid.  Covered: every cluster size, head_dim 64 and 128, bf16 and
fp16, groups of 1 to 8 heads, rows that fill a cluster exactly, rows whose last slice
holds a single key, empty rows, padding CTAs, native-dtype output, the fused append,
a CUDA graph replayed over several calls, and back-to-back calls on one plan.
"""
import numpy as np
import pytest
import torch

import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cl", [2, 4, 8, 16])
@pytest.mark.parametrize("name", ["tiny", "qwen15_mixed", "long_context_b4"])
def test_workloads(name, cl):
    w = W.make(name)
    ro, rl = H.oracle_outputs(w)
    out, lse, info = H.gpu_outputs(w, split_combine=cl)
    assert info["cluster"] == cl and info["num_merge_tasks"] == 0
    H.compare(out, lse, ro, rl, f"{name} cluster {cl}")
    assert pg.read_device_flags() == 0


SHAPES = [(64, 16, "bf16", 14, 2), (128, 16, "fp16", 12, 2), (64, 32, "fp16", 8, 8), (128, 64, "bf16", 16, 2),
          (64, 256, "bf16", 6, 6), (128, 16, "bf16", 8, 1)]


@pytest.mark.parametrize("head_dim,page_size,dtype,hq,hkv", SHAPES)
@pytest.mark.parametrize("cl", [4, 8])
def test_shapes_and_ragged_rows(head_dim, page_size, dtype, hq, hkv, cl):
    """Forced 2-tile slices: rows of exactly cl slices, rows whose last slice is one key,
    empty rows and single-slice rows mixed, so clusters carry holes and padding."""
    tile = 32 if head_dim == 64 else 16
    lens = [cl * 2 * tile, cl * 2 * tile - 1, (cl - 1) * 2 * tile + 1, 0, 1, 2 * tile, 5 * tile + 3, 37]
    w = W.custom("clshape", lens, page_size, hq, hkv, head_dim, dtype, 512, seed=head_dim + page_size + hq + cl)
    ro, rl = H.oracle_outputs(w)
    out, lse, info = H.gpu_outputs(w, split_combine=cl, split_tokens=2 * tile)
    assert info["cluster"] == cl and info["max_splits_used"] == cl
    H.compare(out, lse, ro, rl, f"cluster {cl} d{head_dim} ps{page_size} {dtype} {hq}/{hkv}")
    out16, lse16, _ = H.gpu_outputs(w, torch.bfloat16 if dtype == "bf16" else torch.float16, split_combine=cl,
                                    split_tokens=2 * tile)
    H.compare(out16, lse16, ro, rl, f"cluster {cl} native out", out_dtype=dtype)
    assert pg.read_device_flags() == 0


@pytest.mark.parametrize("stages", [0, 2, 3])
def test_fused_append(stages):
    w = W.custom("clfused", [1200, 33, 700, 4000, 2, 640], 16, 12, 2, 128, "bf16", 1024, seed=21,
                 append_last=True)
    ro, rl = H.oracle_outputs(w)
    dev = H.to_device(w)
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype, max_batch=w.batch,
                   max_q_rows=w.rows, split_combine=8, pipeline_stages=stages)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, kv_indices_host=w.kv_indices)
    out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    plan.append_run(dev["k_new"], dev["v_new"], dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse)
    torch.cuda.synchronize()
    assert plan.info()["cluster"] == 8
    plan.close()
    H.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"cluster fused stages {stages}")
    kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
    import oracle
    oracle.get().kv_append(kp, vp, W.raw16(w.k_new), W.raw16(w.v_new), w.slot_mapping)
    assert np.array_equal(W.raw16(dev["k_pool"]), kp) and np.array_equal(W.raw16(dev["v_pool"]), vp)
    assert pg.read_device_flags() == 0


def test_graph_replay_and_back_to_back_calls():
    """Three calls on one plan, captured in a CUDA graph and replayed twice, each call
    with its own q: the cluster barriers are set up afresh by every launch."""
    w = W.make("qwen15_mixed")
    dev = H.to_device(w)
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype, max_batch=w.batch,
                   max_q_rows=w.rows, split_combine=8)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, kv_indices_host=w.kv_indices)
    gen = torch.Generator().manual_seed(5)
    qs = [torch.randn(w.q.shape, generator=gen).to(w.q.dtype) for _ in range(3)]
    qd = [q.cuda() for q in qs]
    outs = [torch.empty(w.q.shape, dtype=torch.float32, device="cuda") for _ in qs]
    lses = [torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda") for _ in qs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for q, o, l in zip(qd, outs, lses):  # warm-up outside the capture
            plan.run(q, dev["k_pool"], dev["v_pool"], out=o, lse=l, pool_stable=True)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for q, o, l in zip(qd, outs, lses):
            plan.run(q, dev["k_pool"], dev["v_pool"], out=o, lse=l, pool_stable=True)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    plan.close()
    assert pg.read_device_flags() == 0
    for k, q in enumerate(qs):
        w.q = q
        ro, rl = H.oracle_outputs(w)
        H.compare(outs[k].double().cpu().numpy(), lses[k].double().cpu().numpy(), ro, rl, f"graph call {k}")
