"""The CPU oracle against library routines, closed forms and invariants."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("name", sorted(oracle_pins.PINS))
def test_pin(orc, name):
    oracle_pins.PINS[name](orc)


def test_threaded_equals_serial(orc):
    from paged_kv_gqa_05_gb300 import workloads as W
    w = W.custom("thr", [3, 40, 77, 1, 130], 16, 14, 2, 64, "bf16", 64, seed=21)
    o1, l1 = oracle_pins.run(orc, w, nthreads=1)
    o4, l4 = oracle_pins.run(orc, w, nthreads=4)
    assert (o1 == o4).all() and (l1 == l4).all()
