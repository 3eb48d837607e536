"""Shared helpers of the GPU parity tests: run a workload through the C ABI and
through the CPU oracle, and compare element by element."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from paged_kv_gqa_05_gb300 import workloads as W

# Tolerances stated for GPU outputs (bf16/fp16 in, fp32 accumulate) against the
# fp64 oracle on N(0,1) inputs.
MAX_ABS = 5e-3
MEAN_ABS = 5e-4
LSE_ABS = 1e-3

NTHREADS = max(1, min(32, os.cpu_count() or 1))


def oracle_outputs(w: W.Workload, appended: bool = True):
    """Oracle (out, lse) for the workload, after the append of its new rows if any."""
    kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
    orc = oracle.get()
    if appended and w.k_new is not None:
        orc.kv_append(kp, vp, W.raw16(w.k_new), W.raw16(w.v_new), w.slot_mapping)
    return orc.paged_attention(W.raw16(w.q), kp, vp, w.kv_indptr, w.kv_indices, w.last_page_len,
                               w.dtype, qo_indptr=w.qo_indptr, causal=w.causal, nthreads=NTHREADS)


def new_rows_for_query_rows(w: W.Workload, seed: int = 7):
    """One new K/V row per query row: request b's rows land on its last qo_len key
    positions.  Returns (k_new, v_new, flat slots) and NaN-poisons those slots."""
    gen = torch.Generator().manual_seed(seed)
    dt = W.TORCH_DTYPES[w.dtype]
    k_new = torch.randn(w.rows, w.num_kv_heads, w.head_dim, generator=gen).to(dt)
    v_new = torch.randn(w.rows, w.num_kv_heads, w.head_dim, generator=gen).to(dt)
    slots = np.zeros(w.rows, np.int64)
    for b in range(w.batch):
        r0, r1 = (b, b + 1) if w.qo_indptr is None else (int(w.qo_indptr[b]), int(w.qo_indptr[b + 1]))
        n = int(w.kv_lens[b])
        for i, r in enumerate(range(r0, r1)):
            pos = n - (r1 - r0) + i
            page = int(w.kv_indices[w.kv_indptr[b] + pos // w.page_size])
            slots[r] = page * w.page_size + pos % w.page_size
    w.k_pool.view(-1, w.num_kv_heads, w.head_dim)[torch.from_numpy(slots)] = float("nan")
    w.v_pool.view(-1, w.num_kv_heads, w.head_dim)[torch.from_numpy(slots)] = float("nan")
    w.k_new, w.v_new, w.slot_mapping = k_new, v_new, slots
    return k_new, v_new, slots


def to_device(w: W.Workload, device="cuda"):
    d = {
        "q": w.q.to(device),
        "k_pool": w.k_pool.to(device),
        "v_pool": w.v_pool.to(device),
        "kv_indices": torch.from_numpy(w.kv_indices.astype(np.int32)).to(device),
    }
    if w.k_new is not None:
        d["k_new"] = w.k_new.to(device)
        d["v_new"] = w.v_new.to(device)
        d["slot_mapping"] = torch.from_numpy(w.slot_mapping).to(device)
    return d


def gpu_outputs(w: W.Workload, out_dtype=torch.float32, append: bool = True, dev=None,
                host_mirror: bool = True, **plan_opts):
    """Runs (append +) plan + run through the C ABI; returns (out, lse, plan info)."""
    import paged_kv_gqa_05_gb300 as pg
    dev = dev or to_device(w)
    if append and w.k_new is not None:
        pg.kv_append(dev["k_pool"], dev["v_pool"], dev["k_new"], dev["v_new"], dev["slot_mapping"])
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                   max_batch=max(1, w.batch), max_q_rows=max(1, w.rows), **plan_opts)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages,
                qo_indptr=w.qo_indptr, causal=w.causal,
                kv_indices_host=w.kv_indices if host_mirror else None)
    out = torch.empty(dev["q"].shape, dtype=out_dtype, device="cuda")
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse)
    torch.cuda.synchronize()
    info = plan.info()
    plan.close()
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), info


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of |x| in the 16-bit output type."""
    mant = 7 if dtype == "bf16" else 10
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(ax)) - mant - 1)


def compare(out, lse, ref_out, ref_lse, what: str, out_dtype: str = "fp32"):
    """Element-by-element gate; returns (max abs, mean abs) of the output."""
    assert out.shape == ref_out.shape, what
    assert not np.isnan(out).any(), f"{what}: NaN in GPU output (out-of-table read?)"
    err = np.abs(out - ref_out)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if out_dtype == "fp32":
        assert mx <= MAX_ABS, f"{what}: max abs err {mx:.3e} > {MAX_ABS}"
    else:
        bound = MAX_ABS + half_ulp(ref_out, out_dtype)
        worst = float((err - bound).max())
        assert worst <= 0, f"{what}: max abs err exceeds 5e-3 + half-ulp by {worst:.3e}"
    assert mean <= MEAN_ABS, f"{what}: mean abs err {mean:.3e} > {MEAN_ABS}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)), f"{what}: lse finiteness differs"
    if fin.any():
        lerr = float(np.abs(lse[fin] - ref_lse[fin]).max())
        assert lerr <= LSE_ABS, f"{what}: lse err {lerr:.3e}"
    assert np.all(lse[~fin] == ref_lse[~fin]), f"{what}: empty rows must give lse = -inf"
    return mx, mean
