"""CPU-side checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every entry point include/pagedgqa.h declares, and fails with a
status (not a crash) when no device is present."""
import ctypes
import re
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_gqa_05_gb300 import binding, build
    build.build()
    return binding.load()


def declared_entry_points():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = h.read_text()
        names |= set(re.findall(r"PGQA_API\s+[\w\s\*]+?\b(pgqa_\w+)\s*\(", text))
    return names


def test_header_declares_entry_points():
    names = declared_entry_points()
    assert {"pgqa_kv_append", "pgqa_plan_create", "pgqa_plan_update", "pgqa_run",
            "pgqa_plan_destroy"} <= names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_gqa_05_gb300 import binding
    for name in declared_entry_points():
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert set(binding.EXPORTS) == declared_entry_points()


def test_status_strings(lib):
    assert lib.pgqa_abi_version() == 5
    for code in range(7):
        assert lib.pgqa_status_string(code)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour without a device")
def test_no_device_gives_cuda_status(lib):
    from paged_kv_gqa_05_gb300 import binding
    cfg = binding.PlanConfig(14, 2, 64, 16, 0, 4, 4, 0, 0, 0, 0, 0, 0, 0)
    h = ctypes.c_void_p()
    assert lib.pgqa_plan_create(ctypes.byref(h), ctypes.byref(cfg)) == 4
    assert h.value is None
    assert lib.pgqa_last_error()


def test_argument_checks_before_device(lib):
    # shape checks fire before any CUDA call, so they work without a GPU
    cfg_bad = __import__("paged_kv_gqa_05_gb300").binding.PlanConfig(14, 2, 96, 16, 0, 4, 4, 0, 0, 0, 0, 0, 0, 0)
    h = ctypes.c_void_p()
    assert lib.pgqa_plan_create(ctypes.byref(h), ctypes.byref(cfg_bad)) == 2
    assert lib.pgqa_kv_append(None, None, 1, 16, 2, 64, 0, None, None, None, 0, None) == 0
    assert lib.pgqa_kv_append(None, None, 1, 16, 2, 64, 0, None, None, None, 1, None) == 1
    assert lib.pgqa_kv_append(None, None, 1, 12, 2, 64, 0, None, None, None, 1, None) == 2
    assert lib.pgqa_kv_append(None, None, 1, 16, (1 << 20) + 1, 64, 0, None, None, None, 1, None) == 2
    assert lib.pgqa_plan_update(None, None, None, None, 0, None, None, 0, 0, None) == 1
    assert lib.pgqa_run(None, None, None, None, None, 0, None, 0.0, None) == 1
    # RoPE configuration checks, also before any device call
    PC = __import__("paged_kv_gqa_05_gb300").binding.PlanConfig
    assert lib.pgqa_plan_create(ctypes.byref(h), ctypes.byref(PC(14, 2, 64, 16, 0, 4, 4, 0, 0, 0, 0, 0, 0,
                                                                  4096, -1.0))) == 1  # negative theta
    assert lib.pgqa_plan_create(ctypes.byref(h), ctypes.byref(PC(14, 2, 64, 16, 0, 4, 4, 0, 0, 0, 0, 0, 0,
                                                                  0, 1.0e6))) == 1  # no positions
    assert lib.pgqa_plan_create(ctypes.byref(h), ctypes.byref(PC(14, 2, 64, 16, 0, 4, 4, 0, 0, 0, 2, 0, 0,
                                                                  4096, 1.0e6))) == 2  # CUDA-core kernel
    assert lib.pgqa_kv_append_rope(None, None, None, 1, None, None, None, None, 1, None) == 1
    # the static-scratch entry point sizes its scratch without wrapping: 2^30 requests x
    # 2^30 kv heads x 256 slices is a capacity error (the pointers are never dereferenced)
    ptr = 1 << 12
    assert lib.pgqa_decode_static_scratch(ptr, ptr, ptr, ptr, None, 0, ptr, 1 << 30, 1, 16, 1 << 30, 1 << 30,
                                          64, 0, 256, ptr, 0, None, 0.0, None) == 5
    assert lib.pgqa_decode_static_scratch(ptr, ptr, ptr, ptr, None, 0, ptr, 1 << 30, 1, 16, 1 << 30, 1 << 30,
                                          64, 0, 1, ptr, 0, None, 0.0, None) == 5


def test_plan_config_layout():
    """The ctypes mirror of pgqa_plan_config: natural C alignment, rope_theta last."""
    from paged_kv_gqa_05_gb300 import binding
    PC = binding.PlanConfig
    assert PC.max_q_rows.offset == 24 and PC.prefill_splits.offset == 52
    assert PC.rope_max_position.offset == 56 and PC.rope_theta.offset == 64
    assert PC.prefill_kernel.offset == 72 and PC.test_stall_wait_us.offset == 76 and ctypes.sizeof(PC) == 80


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from paged_kv_gqa_05_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load(tmp_path / "missing.so")
