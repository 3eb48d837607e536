"""GPU: the benchmark's timed step in the launch configuration it times -- every
layer's call with the default plan options (fused append where the workload appends;
without new rows, a run() that may load the pools before its dependency wait),
16-bit outputs, all layers replayed from one CUDA graph after a plan update -- checked
against the CPU oracle on layer 0, whose inputs come from the CPU generator."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", ["qwen05_decode", "qwen15_mixed", "long_context_b1", "long_context_b4", "ragged",
                                  "prefill_chunk"])
def test_benchmark_step(name):
    sys.path.insert(0, ROOT)
    import bench
    import paged_kv_gqa_05_gb300 as pg

    device = torch.device("cuda", 0)
    layers = bench.LAYERS[name]
    L = bench.build_layers(name, layers, seed=0, device=device)
    w = L["w"]
    dt = L["q"][0].dtype
    stream = torch.cuda.Stream(device)

    with pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dt, max_batch=w.batch,
                 max_q_rows=w.rows) as plan:
        def update():
            plan.update(w.kv_indptr, w.last_page_len, L["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                        causal=w.causal, stream=stream)

        def calls():
            for l in range(layers):
                if L["slots"] is not None:
                    pg.append_run(plan.handle, L["k_new"][l], L["v_new"][l], L["q"][l], L["k_pool"][l],
                                  L["v_pool"][l], out=L["out"][l], pool_stable=True, stream=stream)
                else:  # no new rows: a run() under the same promise, as the benchmark's step
                    pg.run(plan.handle, L["q"][l], L["k_pool"][l], L["v_pool"][l], out=L["out"][l],
                           pool_stable=True, stream=stream)

        with torch.cuda.stream(stream):
            update()
            calls()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            calls()
        torch.cuda.synchronize()
        L["out"].fill_(float("nan"))
        with torch.cuda.stream(stream):
            for _ in range(3):
                update()
                g.replay()
        torch.cuda.synchronize()
        assert pg.read_device_flags() == 0

    assert not torch.isnan(L["out"]).any(), f"{name}: NaN in a layer's output (out-of-table read?)"
    ro, rl = H.oracle_outputs(w)
    out = L["out"][0].double().cpu().numpy()
    # the benchmark's calls write no lse: the oracle's stands in on both sides
    mx, mean = H.compare(out, rl, ro, rl, f"{name}/benchmark step", out_dtype=w.dtype)
    print(f"{name}: layers={layers} max_abs={mx:.2e} mean_abs={mean:.2e}")
    if L["slots"] is not None:
        # the fused append wrote layer 0's new rows, bit for bit, into its pools
        kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
        oracle.get().kv_append(kp, vp, W.raw16(w.k_new), W.raw16(w.v_new), w.slot_mapping)
        assert np.array_equal(W.raw16(L["k_pool"][0].cpu()), kp), f"{name}: appended K rows differ"
        assert np.array_equal(W.raw16(L["v_pool"][0].cpu()), vp), f"{name}: appended V rows differ"
