"""CPU tests of the plan's host logic through pgqa_plan_schedule (no GPU): the split
heuristic's work lists must cover every admissible key of every (query row, kv head)
exactly once, wire split partials to merges one for one, place each fused-append row
on exactly one CTA, and tile every prefill request's (row, head) pairs and causal key
range; malformed tables fail with the statuses plan_update gives."""
import ctypes
from collections import defaultdict
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import binding as B
from paged_kv_gqa_05_gb300 import workloads as W

SMS = 152


def schedule(w, **options):
    return pg.plan_schedule(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, W.TORCH_DTYPES[w.dtype],
                            w.kv_indptr, w.last_page_len, w.kv_indices, w.num_pages, qo_indptr=w.qo_indptr,
                            causal=w.causal, num_sms=options.pop("num_sms", SMS), **options)


def check_schedule(w, sc, prefill_rows_on_tiles=True):
    """Every invariant of a schedule, derived from the table alone."""
    G = w.num_qo_heads // w.num_kv_heads
    tile = 32 if w.head_dim == 64 else 16
    qo = w.qo_indptr if w.qo_indptr is not None else np.arange(w.batch + 1)
    kv_lens = w.kv_lens.astype(np.int64)
    slices, merges, tiles, info = sc["slices"], sc["merges"], sc["tiles"], sc["info"]
    assert info["num_items"] == len(slices) and info["num_merge_tasks"] == len(merges)
    assert info["num_prefill_tiles"] == len(tiles)
    assert info["total_q_rows"] == int(qo[-1]) and info["kv_tokens"] == int(kv_lens.sum())
    assert info["pipeline_stages"] in (1, 2, 3)

    # launch order: longest slices first
    lens = slices["key_end"] - slices["key_begin"]
    if info["pipeline_stages"] == 1 and len(lens):
        # the wide form: one warp tile per warp (ten warps) unless the caller forced it
        assert G <= 8
    assert np.all(np.diff(lens) <= 0), "slices are not longest-first"
    assert np.all(slices["key_begin"] % tile == 0)

    merge_of = {(int(m["q_row"]), int(m["kv_head"])): m for m in merges}
    assert len(merge_of) == len(merges), "two merges for one (row, kv head)"
    used_slots = set()
    by_pair = defaultdict(list)
    for s in slices:
        by_pair[(int(s["q_row"]), int(s["kv_head"]))].append(s)

    expected_pairs = set()
    merged_pairs = set()
    for b in range(w.batch):
        n, r0, r1 = int(kv_lens[b]), int(qo[b]), int(qo[b + 1])
        L = r1 - r0
        if L > 1 and prefill_rows_on_tiles:
            continue
        for i, r in enumerate(range(r0, r1)):
            a = min(n, max(0, n - L + i + 1)) if w.causal else n
            for kvh in range(w.num_kv_heads):
                expected_pairs.add((r, kvh))
                ss = sorted(by_pair[(r, kvh)], key=lambda s: int(s["key_begin"]))
                assert ss, f"row {r} kv head {kvh} has no slice"
                bounds = [(int(s["key_begin"]), int(s["key_end"])) for s in ss]
                assert bounds[0][0] == 0 and bounds[-1][1] == a, (r, kvh, bounds, a)
                assert all(bounds[j][1] == bounds[j + 1][0] for j in range(len(bounds) - 1)), bounds
                assert all(e > bgn for bgn, e in bounds) or (a == 0 and bounds == [(0, 0)])
                own = n - L + i if L <= n else -1
                writers = [s for s in ss if s["append_pos"] >= 0]
                if own >= 0 and a > 0:
                    assert len(writers) == 1 and int(writers[0]["append_pos"]) == own
                    assert writers[0]["key_begin"] <= own < writers[0]["key_end"] or own >= a
                else:
                    assert not writers
                if len(ss) == 1:
                    assert ss[0]["partial_slot"] == -1 and (r, kvh) not in merge_of
                else:
                    m = merge_of[(r, kvh)]
                    merged_pairs.add((r, kvh))
                    assert int(m["num_splits"]) == len(ss)
                    assert [int(s["partial_slot"]) for s in ss] == list(range(m["slot_base"], m["slot_base"] + len(ss)))
                    for s in ss:
                        assert int(s["partial_slot"]) not in used_slots
                        used_slots.add(int(s["partial_slot"]))
    assert set(by_pair) == expected_pairs, "slices for rows that should have none"
    assert info["max_splits_used"] == max([len(v) for v in by_pair.values()] + [1])

    # prefill tiles: (row, head) pairs of each multi-row request and kv head, key slices of each
    tiles_of = defaultdict(list)
    for t in tiles:
        tiles_of[(int(t["q_row0"]), int(t["kv_head"]), int(t["pair0"]))].append(t)
    seen = set()
    for b in range(w.batch):
        n, r0, r1 = int(kv_lens[b]), int(qo[b]), int(qo[b + 1])
        L = r1 - r0
        if L <= 1 or not prefill_rows_on_tiles:
            continue
        for kvh in range(w.num_kv_heads):
            pairs = None
            m0 = 0
            while m0 < L * G:
                ts = sorted(tiles_of[(r0, kvh, m0)], key=lambda t: int(t["split"]))
                assert ts, f"request {b} kv head {kvh}: no tile at pair {m0}"
                seen.add((r0, kvh, m0))
                pairs = int(ts[0]["pairs"])
                ns = int(ts[0]["num_splits"])
                assert [int(t["split"]) for t in ts] == list(range(ns))
                assert all(int(t["rows"]) == L and int(t["n_keys"]) == n for t in ts)
                i_last = min(L - 1, (m0 + pairs - 1) // G)
                kend = min(n, max(0, n - L + i_last + 1)) if w.causal else n
                bounds = [(int(t["key_begin"]), int(t["key_end"])) for t in ts]
                assert bounds[0][0] == 0 and bounds[-1][1] == kend, (bounds, kend)
                assert all(bounds[j][1] == bounds[j + 1][0] for j in range(ns - 1))
                # slices start on 64-key tiles; trailing ones past a short tile's keys are empty
                assert all(bgn % 64 == 0 or bgn == e == kend for bgn, e in bounds), bounds
                if ns == 1:
                    assert ts[0]["partial_base"] == -1
                else:
                    base = int(ts[0]["partial_base"])
                    assert all(int(t["partial_base"]) == base for t in ts)
                    for i in range(L):
                        m = merge_of[(r0 + i, kvh)]
                        merged_pairs.add((r0 + i, kvh))
                        assert int(m["slot_base"]) == base + i * ns and int(m["num_splits"]) == ns
                m0 += pairs
    assert seen == set(tiles_of), "tiles outside any request's pairs"
    assert merged_pairs == set(merge_of), "merges that no slice or tile feeds"


@pytest.mark.parametrize("name", ["tiny", "qwen05_decode", "qwen15_mixed", "long_context_b1", "long_context_b4",
                                  "ragged", "wide_group", "prefill_chunk"])
def test_workload_schedules(name):
    w = W.make(name)
    sc = schedule(w)
    check_schedule(w, sc)
    again = schedule(w)
    for k in ("slices", "merges", "tiles"):
        assert np.array_equal(sc[k], again[k]), "schedule is not deterministic"


def test_short_rows_fill_one_wave_unsplit():
    """128 requests x 301 keys, 2 kv heads: 256 slices fit the 304 CTA slots of 152 SMs,
    so no row is split, and each row's ten 32-key tiles take the wide form (one warp each)."""
    sc = schedule(W.qwen05_decode())
    assert sc["info"]["num_items"] == 256 and sc["info"]["num_merge_tasks"] == 0
    assert sc["info"]["pipeline_stages"] == 1
    lens = sc["slices"]["key_end"] - sc["slices"]["key_begin"]
    assert lens.max() <= 10 * 32


def test_wide_form_only_for_short_slices_and_narrow_groups():
    """Slices longer than ten warp tiles, and groups of more than 8 heads, keep the ring form."""
    assert schedule(W.make("long_context_b4"))["info"]["pipeline_stages"] in (2, 3)
    assert schedule(W.make("wide_group"))["info"]["pipeline_stages"] in (2, 3)
    assert schedule(W.make("tiny"))["info"]["pipeline_stages"] == 1


def test_long_row_is_spread_over_the_sms():
    """One 32768-key request must be cut into at least one slice per SM."""
    w = W.make("long_context_b1")
    sc = schedule(w)
    assert sc["info"]["num_items"] >= SMS and sc["info"]["num_merge_tasks"] == w.num_kv_heads
    fewer = schedule(w, num_sms=38)
    assert fewer["info"]["num_items"] < sc["info"]["num_items"]
    check_schedule(w, fewer)


@pytest.mark.parametrize("opts", [{"max_splits": 1}, {"split_tokens": 100}, {"split_tokens": 16},
                                  {"pipeline_stages": 2}, {"ctas_per_sm": 3}, {"max_splits": 3},
                                  {"prefill_splits": 1}, {"prefill_splits": 8}, {"prefill_kernel": "mma_sync"}])
def test_options(opts):
    w = W.make("ragged")
    # forced short slices may need more work items than a plan sized for the rows holds
    sc = schedule(w, max_q_rows=8192, **opts)
    check_schedule(w, sc)
    info = sc["info"]
    if opts.get("max_splits") == 1:
        assert info["max_splits_used"] == 1
    if "split_tokens" in opts:
        assert info["split_tokens"] == -(-opts["split_tokens"] // 32) * 32
    if "pipeline_stages" in opts:
        assert info["pipeline_stages"] == 2
    if "prefill_splits" in opts:
        assert set(sc["tiles"]["num_splits"]) == {opts["prefill_splits"]}
    if opts.get("prefill_kernel") == "mma_sync":
        assert set(sc["tiles"]["pairs"]) == {64}


def test_forced_short_slices_over_capacity():
    """Slices forced short enough to outgrow the plan's work list are refused as
    plan_update refuses them."""
    w = W.make("ragged")
    with pytest.raises(B.PagedGQAError) as e:
        schedule(w, split_tokens=32)
    assert e.value.name == "PGQA_ERR_CAPACITY"


@pytest.mark.parametrize("max_batch, max_q_rows", [(10 ** 8, 4), (4, 1 << 24)])
def test_oversized_plan_is_a_capacity_error(max_batch, max_q_rows):
    """Plans whose lists would pass 2^26 entries (the prefill tiles of 10^8 requests, the
    work items of 2^24 rows x 4 kv heads) are refused, not sized from a wrapped count."""
    w = W.custom("cap", [5, 9, 0, 40], 16, 8, 4, 64, "bf16", 8, seed=6)
    with pytest.raises(B.PagedGQAError) as e:
        schedule(w, max_batch=max_batch, max_q_rows=max_q_rows)
    assert e.value.name == "PGQA_ERR_CAPACITY"


def test_cuda_core_kernel_runs_prefill_rows_as_decode_rows():
    """Without tensor-core prefill tiles, every query row of a chunk is a decode row over
    its causal prefix of the keys."""
    w = W.custom("cc", [40, 7, 0, 300], 16, 8, 2, 64, "bf16", 64, seed=3, qo_lens=[5, 1, 1, 3], causal=True)
    sc = schedule(w, decode_kernel="cuda_core", split_tokens=32)
    assert sc["info"]["num_prefill_tiles"] == 0
    check_schedule(w, sc, prefill_rows_on_tiles=False)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_edge_tables(causal, head_dim):
    """Empty requests, one-key requests, a chunk longer than its history, full last pages."""
    w = W.custom("edge", [0, 1, 16, 17, 3, 0, 500], 16, 12, 4, head_dim, "fp16", 128, seed=4,
                 qo_lens=[1, 1, 1, 4, 6, 1, 2], causal=causal)
    for opts in ({}, {"split_tokens": 16}, {"prefill_splits": 3}):
        check_schedule(w, schedule(w, **opts))


def random_table(seed):
    """A seeded page table with the schedule options to plan it under: uniform, equal,
    short and heavy-tailed key counts (empty requests included), some multi-row causal or
    non-causal requests, head shapes, page sizes, split caps, forced prefill key slices,
    slot counts, both kernels and SM counts."""
    rng = np.random.default_rng(5000 + seed)
    hd, ps = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64, 128, 256]))
    hkv, g = int(rng.choice([1, 2, 4, 8])), int(rng.choice([1, 2, 4, 7, 8, 12, 16]))
    batch = int(rng.integers(1, 96))
    mode = rng.random()
    if mode < 0.3:
        lens = rng.integers(0, 5000, batch)
    elif mode < 0.5:
        lens = np.full(batch, int(rng.integers(1, 40000)))
    elif mode < 0.7:
        lens = rng.integers(0, 300, batch)
    else:
        lens = (rng.pareto(1.2, batch) * 500).astype(np.int64).clip(0, 60000)
    qo = None
    if rng.random() < 0.4:
        q = np.ones(batch, np.int64)
        for b in rng.choice(batch, size=max(1, batch // 8), replace=False):
            q[b] = int(rng.integers(2, max(3, min(int(lens[b]) + 4, 700))))
        qo = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
    npg = np.where(lens > 0, -(-lens // ps), 0)
    indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    num_pages = int(indptr[-1]) + 4
    opts = {}
    r = rng.random()
    if r < 0.15:
        opts["max_splits"] = int(rng.integers(1, 6))
    elif r < 0.3:
        opts["prefill_splits"] = int(rng.integers(1, 9))
    if rng.random() < 0.2:
        opts["ctas_per_sm"] = int(rng.integers(1, 4))
    if g <= 8 and rng.random() < 0.1:
        opts["decode_kernel"] = "cuda_core"
    elif rng.random() < 0.2:
        opts["prefill_kernel"] = "mma_sync"
    w = SimpleNamespace(
        num_qo_heads=g * hkv, num_kv_heads=hkv, head_dim=hd, page_size=ps,
        dtype=str(rng.choice(["bf16", "fp16"])), batch=batch, kv_lens=lens.astype(np.int64),
        kv_indptr=indptr, last_page_len=np.where(lens > 0, lens - (npg - 1) * ps, 0).astype(np.int32),
        kv_indices=rng.permutation(num_pages)[: indptr[-1]].astype(np.int32), num_pages=num_pages,
        qo_indptr=qo, causal=qo is not None and bool(rng.random() < 0.7))
    rows = batch if qo is None else int(qo[-1])
    return w, dict(opts, max_q_rows=rows, num_sms=int(rng.choice([152, 148, 132, 76]))), opts


@pytest.mark.parametrize("seed", range(60))
def test_random_tables(seed):
    """Every invariant of the schedule on seeded random tables and options."""
    w, args, opts = random_table(seed)
    sc = schedule(w, **args)
    check_schedule(w, sc, prefill_rows_on_tiles=opts.get("decode_kernel") != "cuda_core")
    if opts.get("max_splits"):
        assert sc["info"]["max_splits_used"] <= opts["max_splits"]


def test_table_errors_match_plan_update():
    w = W.tiny()
    base = dict(kv_indptr=w.kv_indptr, last_page_len=w.last_page_len, kv_indices=w.kv_indices,
                num_pages=w.num_pages)

    def status(**kw):
        args = dict(base, **kw)
        with pytest.raises(B.PagedGQAError) as e:
            pg.plan_schedule(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, torch.bfloat16, **args)
        return e.value.name

    bad = w.kv_indptr.copy()
    bad[0] = 1
    assert status(kv_indptr=bad) == "PGQA_ERR_BAD_PAGE_TABLE"
    last = w.last_page_len.copy()
    last[1] = w.page_size + 1
    assert status(last_page_len=last) == "PGQA_ERR_BAD_PAGE_TABLE"
    idx = w.kv_indices.copy()
    idx[-1] = w.num_pages
    assert status(kv_indices=idx) == "PGQA_ERR_BAD_PAGE_TABLE"
    assert status(kv_indices=np.zeros(0, np.int32)) == "PGQA_ERR_INVALID_ARG"
    assert status(max_batch=1) == "PGQA_ERR_CAPACITY"
    assert status(qo_indptr=np.array([0, 2, 1, 3, 4], np.int32)) == "PGQA_ERR_BAD_PAGE_TABLE"
    with pytest.raises(B.PagedGQAError) as e:
        pg.plan_schedule(w.num_qo_heads, w.num_kv_heads, 96, w.page_size, torch.bfloat16, **base)
    assert e.value.name == "PGQA_ERR_UNSUPPORTED"
    with pytest.raises(B.PagedGQAError) as e:
        pg.plan_schedule(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, torch.bfloat16, num_sms=0, **base)
    assert e.value.name == "PGQA_ERR_INVALID_ARG"
    for stall in (-1, 1000001):  # the failure-path test hook takes 0..1000000 microseconds
        with pytest.raises(B.PagedGQAError) as e:
            pg.plan_schedule(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, torch.bfloat16,
                             test_stall_wait_us=stall, **base)
        assert e.value.name == "PGQA_ERR_INVALID_ARG"


def test_short_output_array_is_a_capacity_error():
    w = W.tiny()
    lib = pg.load()
    cfg = B._config(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, torch.bfloat16, w.batch, w.batch)
    info = B.ScheduleInfo()
    indptr, last, idx = (np.ascontiguousarray(a, np.int32) for a in (w.kv_indptr, w.last_page_len, w.kv_indices))
    p = ctypes.POINTER(ctypes.c_int32)
    args = (ctypes.byref(cfg), SMS, indptr.ctypes.data_as(p), last.ctypes.data_as(p), None, w.batch,
            idx.ctypes.data_as(p), w.num_pages, 0)
    assert lib.pgqa_plan_schedule(*args, None, 0, None, 0, None, 0, ctypes.byref(info)) == 0
    n = info.num_items
    assert n > 1
    short = np.zeros(n - 1, B.SLICE_DTYPE)
    st = lib.pgqa_plan_schedule(*args, short.ctypes.data, n - 1, None, 0, None, 0, ctypes.byref(info))
    assert B.STATUS_NAMES[st] == "PGQA_ERR_CAPACITY" and info.num_items == n
    assert not short.view(np.int32).any(), "nothing is written when the array is too short"


def _mutants(sc):
    """Copies of a schedule, each with one plausible bookkeeping mistake."""
    def copy():
        return {"info": dict(sc["info"]), "slices": sc["slices"].copy(), "merges": sc["merges"].copy(),
                "tiles": sc["tiles"].copy()}
    split = np.flatnonzero(sc["slices"]["partial_slot"] >= 0)
    writer = np.flatnonzero(sc["slices"]["append_pos"] >= 0)
    out = {}
    m = copy()
    m["slices"] = np.delete(m["slices"], split[-1])
    m["info"]["num_items"] -= 1
    out["dropped slice"] = m
    m = copy()
    m["slices"]["key_end"][split[0]] -= 1
    out["short slice"] = m
    m = copy()
    m["slices"]["partial_slot"][split[0]] += 1
    out["wrong partial slot"] = m
    m = copy()
    m["slices"]["append_pos"][writer[0]] -= 1
    out["wrong append position"] = m
    m = copy()
    m["merges"]["num_splits"][0] += 1
    out["wrong merge width"] = m
    m = copy()
    m["tiles"] = np.delete(m["tiles"], 0)
    m["info"]["num_prefill_tiles"] -= 1
    out["dropped tile"] = m
    m = copy()
    m["tiles"]["key_end"][0] += 64
    out["tile past its causal keys"] = m
    return out


@pytest.mark.parametrize("mistake", ["dropped slice", "short slice", "wrong partial slot", "wrong append position",
                                     "wrong merge width", "dropped tile", "tile past its causal keys"])
def test_checker_catches_broken_schedules(mistake):
    """The invariant checker itself fails on each planted mistake."""
    w = W.make("ragged")
    sc = schedule(w)
    check_schedule(w, sc)
    with pytest.raises(AssertionError):
        check_schedule(w, _mutants(sc)[mistake])


def test_prefill_partials_with_many_kv_heads():
    """Split prefill tiles get their partial slots and merges per (request, kv head) for
    any number of kv heads: request 0 (rows 0-1) ends on kv head 512 and request 1
    starts at row 2, kv head 0."""
    w = W.custom("heads513", [20, 30], 16, 513, 513, 64, "bf16", 8, seed=5, qo_lens=[2, 3], causal=True)
    sc = schedule(w, prefill_splits=2)
    assert sc["info"]["num_prefill_tiles"] == 2 * 2 * 513
    check_schedule(w, sc)


def test_prefill_slices_leave_room_for_decode_rows():
    """A chunk alone takes up to two prefill CTAs per SM; beside decode rows about one, so
    that decode CTAs run next to the prefill tiles instead of waiting for them."""
    alone = schedule(W.make("prefill_chunk"))["info"]
    mixed = schedule(W.make("ragged"))["info"]
    assert SMS < alone["num_prefill_tiles"] <= 2 * SMS
    assert mixed["num_items"] > 0 and mixed["num_prefill_tiles"] <= SMS


# The plan's choices for the benchmark's workloads on 152 SMs, each the best or within
# ~1 % of the best of the forced alternatives timed on GB300 (slice length in keys,
# pipeline depth, decode CTAs): a change to the split model shows up here first.
BENCH_CHOICES = {
    "qwen05_decode": (320, 1, 256),      # whole rows, the wide form
    "qwen15_mixed": (448, 3, 292),
    "long_context_b1": (256, 3, 256),    # 128 slices per kv head at three stages
    "long_context_b4": (896, 3, 296),
    "ragged": (2048, 2, 374),            # decode slots net of the 112 prefill CTAs
}


@pytest.mark.parametrize("name", sorted(BENCH_CHOICES))
def test_plan_choices_for_the_benchmark_workloads(name):
    info = schedule(W.make(name))["info"]
    assert (info["split_tokens"], info["pipeline_stages"], info["num_items"]) == BENCH_CHOICES[name]
