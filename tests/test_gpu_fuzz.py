"""GPU: seeded random calls against the CPU oracle.

Each case draws a shape (head_dim, page size, dtype, kv heads, group width), a batch
(lengths from empty to a few thousand keys, some requests with several causal or
non-causal query rows) and plan options (slice length, split cap, pipeline depth or
the wide form, decode and prefill kernels, prefill key slices), then runs the call
through the C ABI and compares every output element and log-sum-exp with the oracle.
Some draws append the step's new rows: inside the call (some of those with the rotary
embedding, the rotated K rows then held to the fp32 rotation's rounding bound, the
other appended rows bit for bit) or by a separate append before it.  The draws cover
combinations the targeted tests do not enumerate.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H
import test_gpu_rope as R

pytestmark = pytest.mark.gpu


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    head_dim = int(rng.choice([64, 128]))
    page_size = int(rng.choice([16, 32, 64, 128, 256]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 12, 16]))
    batch = int(rng.integers(1, 9))
    lens = []
    for _ in range(batch):
        kind = rng.random()
        lens.append(0 if kind < 0.08 else 1 if kind < 0.15 else int(rng.integers(2, 300)) if kind < 0.6
                    else int(rng.integers(300, 3000)))
    multi = rng.random() < 0.4
    qo = None
    if multi:
        qo = [1] * batch
        for b in rng.choice(batch, size=max(1, batch // 3), replace=False):
            if lens[b] >= 2:
                qo[b] = int(rng.integers(2, min(lens[b], 200) + 1))
    causal = bool(rng.random() < 0.7) if multi else False
    tile = 32 if head_dim == 64 else 16
    opts = {}
    r = rng.random()
    if r < 0.3:
        opts["split_tokens"] = tile * int(rng.integers(1, 12))
    elif r < 0.4:
        opts["max_splits"] = int(rng.integers(1, 5))
    kernel = "cuda_core" if (group <= 8 and rng.random() < 0.15) else "tensor_core"
    if kernel == "cuda_core":
        opts["decode_kernel"] = "cuda_core"
    else:
        opts["pipeline_stages"] = int(rng.choice([0, 0, 2, 3] + ([1] if group <= 8 else [])))
    if multi:
        opts["prefill_kernel"] = str(rng.choice(["tcgen05", "mma_sync"]))
        opts["prefill_splits"] = int(rng.integers(0, 5))
    fused = kernel == "tensor_core" and rng.random() < 0.4 and all(q <= n for q, n in zip(qo or [1] * batch, lens))
    out_dtype = "native" if rng.random() < 0.3 else "fp32"
    seed = int(rng.integers(1 << 30))
    rope = fused and bool(rng.random() < 0.5)  # the fused call with the rotary embedding
    # new rows appended by pgqa_kv_append before the call instead of inside it
    separate = (not fused and bool(rng.random() < 0.3) and all(q <= n for q, n in zip(qo or [1] * batch, lens)))
    return dict(head_dim=head_dim, page_size=page_size, dtype=dtype, hkv=hkv, group=group, lens=lens, qo=qo,
                causal=causal, opts=opts, fused=fused, out_dtype=out_dtype, seed=seed, rope=rope, separate=separate)


@pytest.mark.parametrize("seed", range(160))
def test_random_call(seed):
    d = draw(seed)
    hq = d["group"] * d["hkv"]
    pages = sum(-(-n // d["page_size"]) for n in d["lens"]) + 8
    w = W.custom(f"fuzz{seed}", d["lens"], d["page_size"], hq, d["hkv"], d["head_dim"], d["dtype"], pages,
                 seed=d["seed"], qo_lens=d["qo"], causal=d["causal"])
    what = f"fuzz {seed}: {d}"
    if d["fused"] or d["separate"]:
        H.new_rows_for_query_rows(w, seed=seed)
    if d["rope"]:  # q and the new K rows turned at their positions; K pool rows within the rounding bound
        R.check_fused(w, what, **d["opts"])
        return
    ro, rl = H.oracle_outputs(w)
    native = W.TORCH_DTYPES[w.dtype]
    out_dt = native if d["out_dtype"] == "native" else torch.float32
    pg.read_device_flags(clear=True)
    if not d["fused"]:
        out, lse, _ = H.gpu_outputs(w, out_dt, append=d["separate"], **d["opts"])
    else:
        dev = H.to_device(w)
        plan = pg.Plan(hq, d["hkv"], d["head_dim"], d["page_size"], native, max_batch=w.batch,
                       max_q_rows=max(1, w.rows), **d["opts"])
        plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                    causal=w.causal, kv_indices_host=w.kv_indices)
        o = torch.empty(dev["q"].shape, dtype=out_dt, device="cuda")
        l = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
        plan.append_run(dev["k_new"], dev["v_new"], dev["q"], dev["k_pool"], dev["v_pool"], out=o, lse=l)
        torch.cuda.synchronize()
        plan.close()
        out, lse = o.double().cpu().numpy(), l.double().cpu().numpy()
        kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
        oracle.get().kv_append(kp, vp, W.raw16(w.k_new), W.raw16(w.v_new), w.slot_mapping)
        assert np.array_equal(W.raw16(dev["k_pool"]), kp) and np.array_equal(W.raw16(dev["v_pool"]), vp), what
    H.compare(out, lse, ro, rl, what, out_dtype="fp32" if out_dt == torch.float32 else w.dtype)
    assert pg.read_device_flags() == 0, what
