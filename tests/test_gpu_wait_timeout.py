"""GPU: a pipeline wait that can never complete gives up, reports, and leaves the
context usable.

Every barrier wait in the kernels is bounded: after its limit the waiting warp
raises PGQA_FLAG_WAIT_TIMEOUT, lets the copies it did issue land, and the CTA
ends instead of hanging.  The plan option test_stall_wait_us makes one warp of
every decode CTA withhold its first tile's copies, so nothing ever arrives on
that stage's barrier and its wait (limited to the given microseconds) must run
out.  Nothing is in flight into that stage when the wait gives up.  The call
has to return promptly with the flag raised, and a normal call afterwards has
to be correct.
"""
import time

import pytest
import torch

import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

FLAG_WAIT_TIMEOUT = 4


@pytest.mark.parametrize("name", ["tiny", "qwen05_decode"])
def test_withheld_copies_time_out_and_the_next_call_is_right(name):
    w = W.make(name)
    pg.read_device_flags(clear=True)
    t0 = time.perf_counter()
    _, _, info = H.gpu_outputs(w, torch.float32, test_stall_wait_us=1000)
    elapsed = time.perf_counter() - t0
    flags = pg.read_device_flags(clear=True)
    assert flags & FLAG_WAIT_TIMEOUT, f"flags {flags:#x}: the withheld tile's wait did not report"
    assert info["num_items"] > 0
    # one wave of CTAs, each giving up after ~1 ms: far below the default 2 s limit
    assert elapsed < 10.0, f"the stalled call took {elapsed:.1f} s"
    ro, rl = H.oracle_outputs(w)
    out, lse, _ = H.gpu_outputs(w, torch.float32)
    H.compare(out, lse, ro, rl, f"{name} after a timed-out call")
    assert pg.read_device_flags() == 0

