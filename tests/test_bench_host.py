"""CPU tests of bench.py's host logic: the multi-rank plumbing (world size 2 over
gloo: barrier, max/sum over ranks, rank-0-only reporting), the reference arm
(the CPU oracle) JSON line, the ncu traffic lookup and the clock record."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + rank, w)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), w)
    ref = bench.run_reference(bench.main.__globals__["argparse"].Namespace(
        steps=3, warmup=3, workload="tiny", seed=0), r, w)
    q.put((rank, mx, sm, ref is None))
    torch.distributed.destroy_process_group()


def test_two_rank_reductions_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == (0, 2.5, 30.0, False)   # rank 0 times the oracle
    assert got[1] == (1, 2.5, 30.0, True)    # other ranks do no reference work


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--workload", "tiny"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["higher_is_better"] is True and line["steps"] == 3


def test_warmup_floor():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_profiled_traffic_lookup(tmp_path, monkeypatch):
    """The roofline's traffic comes from a committed ncu summary only while the
    summary's source hash matches the kernel's sources; otherwise it is null."""
    sys.path.insert(0, ROOT)
    import bench
    for workload, (name, sources) in bench.PROFILE_FILES.items():
        assert os.path.exists(os.path.join(ROOT, "profiles", name)), name
        assert all(os.path.exists(os.path.join(ROOT, f)) for f in sources)
    assert bench.profiled_traffic("tiny") is None
    # a summary whose hash no longer matches the sources gives no traffic
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "x.md").write_text("traffic_bytes_per_launch: 123\nkernel_sources_sha256_16: 0\n")
    monkeypatch.setattr(bench, "PROFILE_FILES", {"w": ("x.md", bench.DECODE_SOURCES)})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda sources=(): "0")
    assert bench.profiled_traffic("w") == 123
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda sources=(): "1")
    assert bench.profiled_traffic("w") is None


class _Stopped:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_keeps_this_gpu_and_its_throttle_reasons(tmp_path):
    """The clock sampler's summary: only this GPU's rows (by UUID), the median SM clock,
    the highest max clock and every throttle reason seen active."""
    sys.path.insert(0, ROOT)
    import bench
    rows = [
        "GPU-aaaa, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "GPU-bbbb, 600, 2070, 200.0, 0x8, Active, Not Active, Not Active, Not Active",
        "GPU-aaaa, 2010, 2070, 1100.5, 0x4, Not Active, Not Active, Not Active, Active",
        "GPU-aaaa, 1980, 2070, 1010.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "GPU-aaaa, [N/A], 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc, s.path, s.uuid = _Stopped(), str(path), "aaaa"
    rec = s.stop()
    assert rec["sm_mhz"] == 1980.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]  # the other GPU's hw_slowdown is not ours
    assert rec["samples"] == 4 and rec["power_w_max"] == 1100.5
    assert not path.exists()


def test_clock_record_without_samples(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
    path = tmp_path / "clocks.csv"
    path.write_text("GPU-bbbb, 600, 2070, 200.0, 0x8, Active, Not Active, Not Active, Not Active\n"
                    "GPU-cccc, 600, 2070, 200.0, 0x8, Active, Not Active, Not Active, Not Active\n")
    s.proc, s.path, s.uuid = _Stopped(), str(path), "aaaa"
    assert s.stop()["reasons"] == ["no samples for this GPU"]
