"""GPU parity over the supported shape space on small seeded cases: every page
size, both head dims, every group width, both 16-bit types, with kv lengths
that leave ragged tails inside tiles and pages, empty requests, and forced
splits."""
import itertools

import numpy as np
import pytest
import torch

from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

LENS = [0, 1, 5, 16, 17, 31, 33, 100, 257, 700]


KERNELS = ["tensor_core", "cuda_core"]
# tensor-core decode forms: the plan's choice, the wide form (one tile per warp; with
# forced 32-key slices or longer rows it loops on its single stage), and the 2- and 3-stage rings
SCHEDULES = {"auto": {}, "wide": {"pipeline_stages": 1}, "ring2": {"pipeline_stages": 2},
             "ring3": {"pipeline_stages": 3}}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("page_size,head_dim", list(itertools.product([16, 32, 64, 128, 256], [64, 128])))
def test_page_sizes(page_size, head_dim, kernel):
    w = W.custom("sweep", LENS, page_size, 14, 2, head_dim, "bf16", 256, seed=page_size + head_dim)
    ro, rl = H.oracle_outputs(w)
    for opts in ({}, {"split_tokens": 32}, {"max_splits": 1}):
        out, lse, _ = H.gpu_outputs(w, decode_kernel=kernel, **opts)
        H.compare(out, lse, ro, rl, f"{kernel}/ps{page_size}/d{head_dim}/{opts}")


@pytest.mark.parametrize("schedule", sorted(SCHEDULES))
@pytest.mark.parametrize("head_dim,dtype", [(64, "bf16"), (128, "fp16")])
def test_decode_schedules(schedule, head_dim, dtype):
    w = W.custom("sched", LENS * 3, 16, 14, 2, head_dim, dtype, 512, seed=head_dim + 5)
    ro, rl = H.oracle_outputs(w)
    for opts in ({}, {"split_tokens": 32}):
        out, lse, _ = H.gpu_outputs(w, **SCHEDULES[schedule], **opts)
        H.compare(out, lse, ro, rl, f"{schedule}/d{head_dim}/{opts}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("group,dtype,head_dim",
                         list(itertools.product([1, 2, 3, 4, 5, 6, 7, 8], ["bf16", "fp16"], [64, 128])))
def test_groups(group, dtype, head_dim, kernel):
    hkv = 2 if group <= 4 else 1
    w = W.custom("grp", [3, 40, 129, 300], 16, group * hkv, hkv, head_dim, dtype, 64,
                 seed=group * 7 + head_dim)
    ro, rl = H.oracle_outputs(w)
    out, lse, _ = H.gpu_outputs(w, split_tokens=64, decode_kernel=kernel)
    H.compare(out, lse, ro, rl, f"{kernel}/g{group}/{dtype}/d{head_dim}")


@pytest.mark.parametrize("group,dtype,head_dim",
                         [(g, dt, d) for g in range(9, 17) for dt, d in (("bf16", 64), ("fp16", 128))] +
                         [(16, "fp16", 64), (12, "bf16", 128)])
@pytest.mark.parametrize("stages", [2, 3])
def test_wide_groups(group, dtype, head_dim, stages):
    """9..16 query heads per kv head: the tensor-core tile's second 8-head n tile."""
    w = W.custom("wgrp", [3, 40, 129, 300, 1000], 16, group * 2, 2, head_dim, dtype, 128,
                 seed=group * 5 + head_dim + stages)
    ro, rl = H.oracle_outputs(w)
    out, lse, _ = H.gpu_outputs(w, split_tokens=64, pipeline_stages=stages)
    H.compare(out, lse, ro, rl, f"wide g{group}/{dtype}/d{head_dim}/st{stages}")


def test_wide_form_is_refused_for_wide_groups():
    """The wide decode form serves groups of up to 8 heads; asked for with 16 it is refused."""
    import paged_kv_gqa_05_gb300 as pg
    with pytest.raises(pg.PagedGQAError) as e:
        pg.Plan(32, 2, 128, 16, torch.bfloat16, max_batch=1, max_q_rows=1, pipeline_stages=1)
    assert e.value.name == "PGQA_ERR_UNSUPPORTED"


def test_all_empty_batch():
    w = W.custom("empty", [0, 0, 0], 16, 4, 2, 64, "bf16", 4, seed=1)
    out, lse, _ = H.gpu_outputs(w)
    assert not out.any() and np.all(lse == -np.inf)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("causal", [True, False])
def test_multi_row_requests(causal, kernel):
    """Ragged rows (qo_indptr) with and without the bottom-right causal mask."""
    w = W.custom("rag", [40, 7, 300, 64], 16, 14, 2, 64, "bf16", 64, seed=11,
                 qo_lens=[13, 1, 5, 64], causal=causal)
    ro, rl = H.oracle_outputs(w)
    out, lse, _ = H.gpu_outputs(w, split_tokens=64, decode_kernel=kernel)
    H.compare(out, lse, ro, rl, f"ragged causal={causal}")


@pytest.mark.parametrize("head_dim,n,kernel", [(64, 20000, "tensor_core"), (128, 12000, "tensor_core"),
                                                (128, 9000, "cuda_core")])
def test_block_merge_long_slice_lists(head_dim, n, kernel):
    """One-tile slices of one long row: 500-750 slices per (row, kv head), beyond the
    block merge's up-front requests (256 per thread group), so its loop over the rest runs;
    an empty row and a short one ride along."""
    tile = 32 if head_dim == 64 else 16
    w = W.custom("longlist", [n, 0, 40], 64, 8, 2, head_dim, "bf16", n // 64 + 16, seed=n + head_dim)
    ro, rl = H.oracle_outputs(w)
    out, lse, info = H.gpu_outputs(w, split_tokens=tile, decode_kernel=kernel)
    assert info["max_splits_used"] > 256
    H.compare(out, lse, ro, rl, f"{info['max_splits_used']} slices d{head_dim} {kernel}")


def test_many_short_rows():
    """4096 decode rows of 0-64 keys: a grid of 8192 unsplit CTAs, many waves deep."""
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(0, 65, 4096)]
    w = W.custom("many", lens, 16, 14, 2, 64, "bf16", sum(-(-n // 16) for n in lens) + 16, seed=5)
    ro, rl = H.oracle_outputs(w)
    out, lse, info = H.gpu_outputs(w)
    assert info["num_items"] == 8192 and info["num_merge_tasks"] == 0
    H.compare(out, lse, ro, rl, "4096 short rows")


def test_explicit_scale():
    import oracle
    import paged_kv_gqa_05_gb300 as pg
    w = W.custom("scale", [50, 77], 16, 8, 2, 128, "fp16", 32, seed=3)
    ro, rl = oracle.get().paged_attention(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool),
                                          w.kv_indptr, w.kv_indices, w.last_page_len, "fp16",
                                          scale=0.3)
    dev = H.to_device(w)
    plan = pg.Plan(8, 2, 128, 16, torch.float16, 2, 2)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages)
    lse = torch.empty(2, 8, device="cuda")
    out = plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out_dtype=torch.float32, lse=lse,
                   sm_scale=0.3)
    H.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "scale 0.3")


@pytest.mark.parametrize("group,head_dim,page_size,dtype",
                         [(7, 64, 64, "bf16"), (6, 128, 256, "fp16"), (1, 64, 16, "bf16"), (8, 128, 32, "bf16"),
                          (3, 64, 128, "fp16"), (5, 128, 16, "bf16"), (16, 64, 64, "bf16"),
                          (12, 128, 16, "fp16")])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("prefill_kernel", ["tcgen05", "mma_sync"])
def test_prefill_segments(group, head_dim, page_size, dtype, causal, prefill_kernel):
    """Chunks of query rows (tensor-core prefill tiles) mixed with decode rows,
    chunk lengths not multiples of 64 / G, plus a chunk longer than its history
    (its first rows have no admissible key under the causal mask)."""
    hkv = 2 if group <= 4 else 1
    lens = [300, 5, 1030, 77, 3]
    qo = [70, 1, 200, 77, 5]
    w = W.custom("pf", lens, page_size, group * hkv, hkv, head_dim, dtype, 128, seed=group + head_dim,
                 qo_lens=qo, causal=causal)
    ro, rl = H.oracle_outputs(w)
    out, lse, info = H.gpu_outputs(w, prefill_kernel=prefill_kernel)
    assert info["num_prefill_tiles"] > 0
    H.compare(out, lse, ro, rl, f"prefill/{prefill_kernel} g{group} d{head_dim} ps{page_size} {dtype} causal={causal}")


@pytest.mark.gpu
@pytest.mark.parametrize("prefill_kernel", ["tcgen05", "mma_sync"])
@pytest.mark.parametrize("splits", [1, 2, 3, 8])
def test_prefill_key_slices_repeated(prefill_kernel, splits):
    """A fixed number of key slices per prefill tile (1, 2, 3 and the maximum 8), their
    partials merged by the merge kernel.  The same plan runs five times, the last
    three from one CUDA graph, each output checked against the oracle: nothing a call
    leaves in the plan's buffers may change the next one."""
    import paged_kv_gqa_05_gb300 as pg
    w = W.custom("slices", [1536, 40, 700], 64, 14, 2, 64, "bf16", 128, seed=11 + splits,
                 qo_lens=[300, 1, 129], causal=True)
    ro, rl = H.oracle_outputs(w)
    dev = H.to_device(w)
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dev["q"].dtype,
                   max_batch=w.batch, max_q_rows=w.rows, prefill_kernel=prefill_kernel, prefill_splits=splits)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                causal=True, kv_indices_host=w.kv_indices)
    info = plan.info()
    assert info["num_prefill_tiles"] > 0
    assert (info["num_merge_tasks"] > 0) == (splits > 1)
    out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    for _ in range(2):
        out.fill_(float("nan"))
        plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse)
        torch.cuda.synchronize()
        H.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
                  f"{prefill_kernel} {splits} slices, eager")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        H.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
                  f"{prefill_kernel} {splits} slices, graph")
    plan.close()


@pytest.mark.gpu
@pytest.mark.parametrize("prefill_kernel", ["tcgen05", "mma_sync"])
@pytest.mark.parametrize("head_dim,group", [(64, 7), (128, 6)])
def test_prefill_growing_scores(prefill_kernel, head_dim, group):
    """Keys scaled up tile by tile (x(1 + 3 t) for the 64-key tile t of each request), so
    a row's maximum jumps far past its running maximum again and again: this drives the
    tcgen05 kernel's rescale of O in tensor memory on many tiles (random scores seldom
    move the maximum by the 2^8 that triggers it), and the mma.sync kernel's online
    rescale alike."""
    w = W.custom("grow", [1100, 300, 70], 64, group, 1, head_dim, "bf16", 64, seed=5 + head_dim,
                 qo_lens=[260, 1, 70], causal=True)
    ps = w.page_size
    for b in range(w.batch):
        p0, p1 = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        n = (p1 - p0 - 1) * ps + int(w.last_page_len[b]) if p1 > p0 else 0
        for j in range(n):
            page = int(w.kv_indices[p0 + j // ps])
            w.k_pool[page, j % ps] = (w.k_pool[page, j % ps].float() * (1 + 3 * (j // 64))).to(w.k_pool.dtype)
    ro, rl = H.oracle_outputs(w)
    out, lse, info = H.gpu_outputs(w, prefill_kernel=prefill_kernel)
    assert info["num_prefill_tiles"] > 0
    H.compare(out, lse, ro, rl, f"growing scores {prefill_kernel} d{head_dim} g{group}")


@pytest.mark.gpu
@pytest.mark.parametrize("prefill_kernel", ["tcgen05", "mma_sync"])
def test_long_chunk_sampled_rows(prefill_kernel):
    """The suite's largest prefill launch: one 3000-row causal chunk over 4000 keys
    (d 128, g 8, page 64; 375 tiles of 64 or 188 of 128 (row, head) pairs per kv head
    before key slicing), checked on sampled (row, head) pairs that the oracle computes
    one by one: the first rows, the last row and random ones, across both kv heads."""
    import oracle
    w = W.custom("long_chunk", [4000], 64, 16, 2, 128, "bf16", 80, seed=31, qo_lens=[3000], causal=True)
    out, lse, info = H.gpu_outputs(w, prefill_kernel=prefill_kernel)
    assert info["num_prefill_tiles"] > 0
    orc = oracle.get()
    rng = np.random.default_rng(7)
    rows = [0, 1, 2, 1499, 2999] + [int(x) for x in rng.integers(0, 3000, 8)]
    for r in rows:
        for h in (0, 5, 7, 8, 13, 15):
            o, l = orc.attention_partial(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool), w.kv_indptr,
                                         w.kv_indices, w.last_page_len, w.dtype, 0, r, h, 0, 4000,
                                         qo_indptr=w.qo_indptr, causal=True)
            assert np.abs(out[r, h] - o).max() <= H.MAX_ABS, (prefill_kernel, r, h)
            assert abs(lse[r, h] - l) <= H.LSE_ABS, (prefill_kernel, r, h)


@pytest.mark.gpu
def test_zero_sized_calls():
    """Empty calls are accepted and do nothing: an append of zero tokens (plain and
    rotating), and a plan over zero requests run on zero query rows."""
    import paged_kv_gqa_05_gb300 as pg
    g = torch.Generator(device="cuda").manual_seed(3)
    k_pool = torch.randn(4, 16, 2, 64, device="cuda", generator=g).to(torch.bfloat16)
    v_pool = torch.randn(4, 16, 2, 64, device="cuda", generator=g).to(torch.bfloat16)
    before_k, before_v = k_pool.clone(), v_pool.clone()
    empty = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.empty(0, dtype=torch.int64, device="cuda")
    pg.kv_append(k_pool, v_pool, empty, empty, slots)
    with pg.Plan(14, 2, 64, 16, torch.bfloat16, max_batch=4, max_q_rows=4, rope_theta=1e6,
                 rope_max_position=64) as plan:
        plan.kv_append_rope(k_pool, v_pool, empty, empty, slots, torch.empty(0, dtype=torch.int32, device="cuda"))
        plan.update(np.zeros(1, np.int32), np.zeros(0, np.int32), torch.empty(0, dtype=torch.int32, device="cuda"), 4)
        info = plan.info()
        assert info["num_items"] == 0 and info["num_prefill_tiles"] == 0 and info["total_q_rows"] == 0
        out = plan.run(torch.empty(0, 14, 64, dtype=torch.bfloat16, device="cuda"), k_pool, v_pool)
        assert out.shape == (0, 14, 64)
    torch.cuda.synchronize()
    assert torch.equal(k_pool, before_k) and torch.equal(v_pool, before_v)
    assert pg.read_device_flags() == 0

