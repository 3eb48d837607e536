"""GPU parity of the full path (append + plan + split-KV partial + merge) against
the CPU fp64 oracle, on the five seeded workloads at full size."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

_cache = {}


def _ref(name):
    if name not in _cache:
        w = W.make(name)
        _cache[name] = (w, H.oracle_outputs(w))
    return _cache[name]


@pytest.mark.parametrize("name", ["tiny", "qwen05_decode", "qwen15_mixed", "long_context_b1",
                                  "long_context_b4", "ragged"])
def test_workload_fp32_out(name):
    w, (ro, rl) = _ref(name)
    out, lse, info = H.gpu_outputs(w, torch.float32)
    mx, mean = H.compare(out, lse, ro, rl, name)
    print(f"{name}: items={info['num_items']} merges={info['num_merge_tasks']} "
          f"split={info['split_tokens']} max_abs={mx:.2e} mean_abs={mean:.2e}")
    # fp32 accumulation leaves far more room than the gate; a regression shows here first
    assert mx < 1e-4, f"{name}: fp32 path error {mx:.2e} is larger than fp32 arithmetic explains"


@pytest.mark.parametrize("name", ["tiny", "qwen05_decode", "qwen15_mixed", "long_context_b1", "ragged"])
def test_workload_cuda_core_kernel(name):
    """The CUDA-core (fp32 FMA) decode kernel on the same workloads."""
    w, (ro, rl) = _ref(name)
    out, lse, _ = H.gpu_outputs(w, torch.float32, decode_kernel="cuda_core")
    H.compare(out, lse, ro, rl, name + "/cuda_core")


@pytest.mark.parametrize("name", ["tiny", "qwen05_decode", "qwen15_mixed", "ragged"])
def test_workload_native_out(name):
    w, (ro, rl) = _ref(name)
    dt = W.TORCH_DTYPES[w.dtype]
    out, lse, _ = H.gpu_outputs(w, dt)
    H.compare(out, lse, ro, rl, name + "/" + w.dtype, out_dtype=w.dtype)


@pytest.mark.parametrize("name", ["tiny", "qwen05_decode", "long_context_b1"])
def test_split_vs_unsplit_same_pages(name):
    """Both decode schedules on the same pages: never split, and split into
    many short slices merged by log-sum-exp."""
    w, (ro, rl) = _ref(name)
    dev = H.to_device(w)
    import paged_kv_gqa_05_gb300 as pg
    if w.k_new is not None:
        pg.kv_append(dev["k_pool"], dev["v_pool"], dev["k_new"], dev["v_new"], dev["slot_mapping"])
    o1, l1, i1 = H.gpu_outputs(w, append=False, dev=dev, max_splits=1)
    o2, l2, i2 = H.gpu_outputs(w, append=False, dev=dev, split_tokens=64)
    assert i1["num_merge_tasks"] == 0 and i1["max_splits_used"] == 1
    if int(w.kv_lens.max()) > 64:
        assert i2["num_merge_tasks"] > 0
    H.compare(o1, l1, ro, rl, name + "/unsplit")
    H.compare(o2, l2, ro, rl, name + "/split64")
    assert np.abs(o1 - o2).max() < 1e-4


def test_deterministic():
    w, _ = _ref("qwen15_mixed")
    dev = H.to_device(w)
    a = H.gpu_outputs(w, dev=dev)
    b = H.gpu_outputs(w, dev=dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_no_host_mirror_same_result():
    w, (ro, rl) = _ref("tiny")
    out, lse, _ = H.gpu_outputs(w, host_mirror=False)
    H.compare(out, lse, ro, rl, "tiny/no-mirror")


def test_sampled_rows_full_size_long_context_b4():
    """Full-size launch as the benchmark runs it, checked on sampled rows/heads
    the oracle computes one by one."""
    import oracle
    w, _ = _ref("long_context_b4")
    out, lse, info = H.gpu_outputs(w, torch.bfloat16)
    orc = oracle.get()
    rng = np.random.default_rng(5)
    for _ in range(6):
        b = int(rng.integers(w.batch))
        h = int(rng.integers(w.num_qo_heads))
        o, l = orc.attention_partial(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool),
                                     w.kv_indptr, w.kv_indices, w.last_page_len, w.dtype,
                                     b, b, h, 0, int(w.kv_lens[b]))
        err = np.abs(out[b, h] - o) - H.half_ulp(o, "bf16")
        assert err.max() <= H.MAX_ABS
        assert abs(lse[b, h] - l) <= H.LSE_ABS
    assert info["num_merge_tasks"] > 0


@pytest.mark.parametrize("kernel_opts", [{}, {"pipeline_stages": 2}, {"decode_kernel": "cuda_core"}],
                         ids=["per-item", "two-stage", "cuda-core"])
def test_split_rows_repeated_calls(kernel_opts):
    """128-token slices (6 to 24 per row) on each decode kernel, merged by the merge
    kernel.  The same plan runs three times eagerly and twice from a CUDA graph, each
    output checked against the oracle: nothing a call leaves in the plan's buffers may
    change the next one."""
    import paged_kv_gqa_05_gb300 as pg
    w = W.custom("splits", [1, 50, 700, 1500, 2048, 3000], 16, 14, 2, 64, "bf16", 640, seed=21,
                 append_last=True)
    ro, rl = H.oracle_outputs(w)
    dev = H.to_device(w)
    pg.kv_append(dev["k_pool"], dev["v_pool"], dev["k_new"], dev["v_new"], dev["slot_mapping"])
    with pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                 max_batch=w.batch, max_q_rows=w.rows, split_tokens=128, **kernel_opts) as plan:
        plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, kv_indices_host=w.kv_indices)
        info = plan.info()
        # split rows: 700, 1500, 2048 and 3000 keys (6, 12, 16, 24 slices), two kv heads each
        assert info["num_merge_tasks"] == 2 * 4 and info["max_splits_used"] == 24
        out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
        lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
        for _ in range(3):
            out.fill_(float("nan"))
            plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse)
            torch.cuda.synchronize()
            H.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"splits {kernel_opts}")
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse)
        for _ in range(2):
            out.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            H.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"splits {kernel_opts} graph")
    assert pg.read_device_flags() == 0


@pytest.mark.parametrize("name", ["tiny", "qwen15_mixed", "long_context_b1", "ragged"])
def test_pool_stable_run_is_the_plain_run(name):
    """pgqa_append_run without new rows and with PGQA_RUN_POOL_STABLE (the loads may start
    before the dependency wait) gives the plain run()'s result bit for bit, and the oracle's."""
    import paged_kv_gqa_05_gb300 as pg
    w, (ro, rl) = _ref(name)
    dev = H.to_device(w)
    if w.k_new is not None:
        pg.kv_append(dev["k_pool"], dev["v_pool"], dev["k_new"], dev["v_new"], dev["slot_mapping"])
    with pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                 max_batch=w.batch, max_q_rows=w.rows) as plan:
        plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                    causal=w.causal)
        res = []
        for stable in (False, True):
            out = torch.full(dev["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full(dev["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
            plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse, pool_stable=stable)
            torch.cuda.synchronize()
            res.append((out.double().cpu().numpy(), lse.double().cpu().numpy()))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
    H.compare(res[1][0], res[1][1], ro, rl, name + "/pool-stable run")
