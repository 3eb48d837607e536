"""CPU checks of the binding's argument checks.  With the library calls replaced by
recorders: Plan.run and Plan.append_run refuse tensors smaller than what the plan's
last successful update reads or writes through them, before anything is launched.
Through pgqa_plan_schedule: host page-table arrays are converted to int32 only when
every value fits."""
import pytest
import torch

from paged_kv_gqa_05_gb300 import binding as B

HQ, HKV, D, PS, PAGES, ROWS = 4, 2, 64, 16, 6, 3


@pytest.fixture
def plan(monkeypatch):
    calls = []
    monkeypatch.setattr(B, "plan_update", lambda *a, **k: calls.append(("update", a, k)))
    monkeypatch.setattr(B, "run", lambda *a, **k: calls.append(("run", a, k)))
    monkeypatch.setattr(B, "append_run", lambda *a, **k: calls.append(("append_run", a, k)))
    p = object.__new__(B.Plan)
    p.handle = 1234
    p._shape(HQ, HKV, D, PS)
    p.info = lambda: {"total_q_rows": ROWS}
    p.calls = calls
    yield p
    p.handle = None  # not a real plan: nothing for close() to destroy


def t(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def pools(pages=PAGES):
    return t(pages, PS, HKV, D), t(pages, PS, HKV, D)


def test_no_check_before_a_successful_update(plan):
    k, v = pools(1)
    plan.run(t(1, HQ, D), k, v)  # the library refuses a plan without an update itself
    assert plan.calls[-1][0] == "run"


def test_full_sized_tensors_pass(plan):
    plan.update([0, 1, 2, 3], [1, 1, 1], t(3), PAGES, qo_indptr=None)
    k, v = pools()
    plan.run(t(ROWS, HQ, D), k, v, out=torch.zeros(ROWS, HQ, D), lse=torch.zeros(ROWS, HQ))
    plan.run(t(ROWS + 5, HQ, D), k, v)  # larger is fine
    plan.append_run(t(ROWS, HKV, D), t(ROWS, HKV, D), t(ROWS, HQ, D), k, v)
    plan.append_run(k_new=t(ROWS, HKV, D), v_new=t(ROWS, HKV, D), q=t(ROWS, HQ, D), k_pool=k, v_pool=v)
    assert [c[0] for c in plan.calls] == ["update", "run", "run", "append_run", "append_run"]
    assert all(c[1][0] == 1234 for c in plan.calls)


@pytest.mark.parametrize("which", ["q", "out", "lse", "k_pool", "v_pool"])
def test_run_refuses_short_tensors(plan, which):
    plan.update([0, 1, 2, 3], [1, 1, 1], t(3), PAGES)
    k, v = pools()
    args = dict(q=t(ROWS, HQ, D), k_pool=k, v_pool=v, out=torch.zeros(ROWS, HQ, D), lse=torch.zeros(ROWS, HQ))
    args[which] = args[which][:-1]  # one row or page short
    n = len(plan.calls)
    with pytest.raises(ValueError, match=which):
        plan.run(**args)
    assert len(plan.calls) == n, "nothing reaches the library"


@pytest.mark.parametrize("which", ["k_new", "v_new", "q", "k_pool"])
def test_append_run_refuses_short_tensors(plan, which):
    plan.update([0, 1, 2, 3], [1, 1, 1], t(3), PAGES)
    k, v = pools()
    args = [t(ROWS, HKV, D), t(ROWS, HKV, D), t(ROWS, HQ, D), k, v]
    names = ["k_new", "v_new", "q", "k_pool", "v_pool"]
    i = names.index(which)
    args[i] = args[i][:-1]
    with pytest.raises(ValueError, match=which):
        plan.append_run(*args)


def test_failed_update_turns_the_checks_off(plan, monkeypatch):
    plan.update([0, 1, 2, 3], [1, 1, 1], t(3), PAGES)

    def refuse(*a, **k):
        raise B.PagedGQAError(3, "malformed page table")

    monkeypatch.setattr(B, "plan_update", refuse)
    with pytest.raises(B.PagedGQAError):
        plan.update([0, 1], [1], t(1), 1)
    k, v = pools(1)
    plan.run(t(1, HQ, D), k, v)  # passed on: the library reports the plan as not updated
    assert plan.calls[-1][0] == "run"


@pytest.mark.parametrize("bad", [[0, 1 << 31], [-(1 << 31) - 1], [0.5, 1.0], [True, False]])
def test_host_tables_are_not_truncated(bad):
    """Page-table arrays that int32 cannot hold exactly are refused, not wrapped."""
    with pytest.raises(ValueError):
        B.plan_schedule(4, 2, 64, 16, torch.bfloat16, bad, [1], [0], 4)


def test_host_tables_accept_any_integer_type():
    import numpy as np
    for a in ([0, 1], np.array([0, 1], np.int64), torch.tensor([0, 1]), np.array([0, 1], np.uint16)):
        s = B.plan_schedule(4, 2, 64, 16, torch.bfloat16, a, [5], [0], 4)
        assert s["info"]["num_items"] == 2


def test_append_needs_a_slot_per_row():
    k = torch.zeros(3, HKV, D, dtype=torch.bfloat16)
    kp, vp = pools()
    with pytest.raises(ValueError, match="one slot per row"):
        B.kv_append(kp, vp, k, k, torch.zeros(2, dtype=torch.int64))


@pytest.mark.parametrize("which", ["kv_indptr", "last_page_len", "out", "lse"])
def test_static_scratch_needs_full_tables(which):
    q = t(ROWS, HQ, D)
    kp, vp = pools()
    args = dict(kv_indptr=torch.zeros(ROWS + 1, dtype=torch.int32), kv_indices=torch.zeros(0, dtype=torch.int32),
                last_page_len=torch.zeros(ROWS, dtype=torch.int32), out=torch.zeros(ROWS, HQ, D),
                lse=torch.zeros(ROWS, HQ))
    args[which] = args[which][:-1]
    with pytest.raises(ValueError, match=which):
        B.decode_static_scratch(q, kp, vp, splits=2, **args)


@pytest.mark.parametrize("which", ["out", "lse", "q"])
def test_module_run_checks_outputs_against_q(which):
    """The bare-handle calls cannot see the plan, but out and lse must cover q."""
    q, out, lse = t(ROWS, HQ, D), torch.zeros(ROWS, HQ, D), torch.zeros(ROWS, HQ)
    if which == "out":
        out = out[:-1]
    elif which == "lse":
        lse = lse[:-1]
    else:
        q = q.reshape(ROWS, HQ * D)
    kp, vp = pools()
    with pytest.raises(ValueError, match=which):
        B.run(1234, q, kp, vp, out=out, lse=lse)
    with pytest.raises(ValueError, match=which):
        B.append_run(1234, t(ROWS, HKV, D), t(ROWS, HKV, D), q, kp, vp, out=out, lse=lse)
