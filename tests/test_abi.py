"""The C-ABI library builds for sm_103a, loads, and exports every entry point that
include/rkv.h declares; host-only calls validate arguments without a GPU."""
import ctypes
import os
import re

import pytest
import torch

from reference_residual_kv_gb300 import build, rkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "rkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(rkv_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return rkv.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("rkv_build_ref_pool", "rkv_compress", "rkv_gather_dequant", "rkv_query_sizes"):
        assert n in names
    assert set(names) == set(rkv.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_query_sizes_host_only(lib):
    p = rkv.make_params(32, 1, 8192, 8, 128, 1024, 512, stride=8)
    assert rkv.rkv_n_ref(p) == 1024
    pool, cache, ws = rkv.rkv_query_sizes(p)
    assert cache == 32 * 8192 * (256 + 16 * 8 + 16)
    assert pool == 1024 * 4 + 2 * 8192 * 4 + 32 * 1024 * 2048 * 2 + 32 * 1024 * 4
    assert ws > 0
    p8 = rkv.make_params(1, 1, 131072, 8, 128, 1024, 512, stride=16, ref_dtype="fp8")
    assert rkv.rkv_n_ref(p8) == 8192
    assert rkv.rkv_query_sizes(p8)[0] == 8192 * 4 + 2 * 131072 * 4 + 8192 * 2048 + 8192 * 4


@pytest.mark.parametrize("field,value,code", [
    ("bits", 3, rkv.RKV_ERR_INVALID_ARG),
    ("T", 0, rkv.RKV_ERR_INVALID_ARG),
    ("stride", 0, rkv.RKV_ERR_INVALID_ARG),
    ("k", 5, rkv.RKV_ERR_UNSUPPORTED),
    ("group", 16, rkv.RKV_ERR_UNSUPPORTED),
    ("d_c", 48, rkv.RKV_ERR_UNSUPPORTED),
    ("ref_dtype", rkv.RKV_FP8_E4M3, rkv.RKV_ERR_INVALID_ARG),   # FP8 refs need bf16 kv
])
def test_invalid_params_rejected_before_any_launch(lib, field, value, code):
    p = rkv.make_params(1, 1, 256, 2, 64, 256, 64, kv_dtype="f32")
    setattr(p, field, value)
    a = ctypes.c_size_t()
    assert lib.rkv_query_sizes(ctypes.byref(p), ctypes.byref(a), None, None) == code
    pool = rkv.rkv_ref_pool(16, 16, 16, 16, 16)
    # validation fails before anything touches the device (no GPU here)
    assert lib.rkv_build_ref_pool(ctypes.byref(p), 16, ctypes.byref(pool), None) == code


def test_null_and_misaligned_pointers_rejected(lib):
    p = rkv.make_params(1, 1, 256, 2, 64, 256, 64, kv_dtype="f32")
    pool = rkv.rkv_ref_pool(16, 16, 16, 16, 16)
    assert lib.rkv_build_ref_pool(ctypes.byref(p), None, ctypes.byref(pool), None) == rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_build_ref_pool(ctypes.byref(p), 24, ctypes.byref(pool), None) == rkv.RKV_ERR_ALIGNMENT
    cache = rkv.rkv_cache(16, 16, 16)
    st = lib.rkv_compress(ctypes.byref(p), 16, ctypes.byref(pool), 16, 16, 16, ctypes.byref(cache),
                          None, 0, None, 16, None)
    assert st == rkv.RKV_ERR_WORKSPACE
    st = lib.rkv_gather_dequant(ctypes.byref(p), ctypes.byref(pool), ctypes.byref(cache), 16, 4,
                                16, 16, 7, 16, None)
    assert st == rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_status_string(rkv.RKV_ERR_INDEX) == b"index out of range (device)"


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rkv, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rkv, "_lib", None)
    with pytest.raises(RuntimeError):
        rkv.lib()


def test_dynamic_schedule_counts_host_side(lib):
    # rkv_n_ref follows the dynamic recurrence [RKV §2.6]; under the Table VI reading
    # (s0 = 10, n_sink = 0, 261888 scheduled positions) it gives the table's counts
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "table6_ref_counts.json")))
    for alpha, n in zip(g["alpha"], g["n_ref"]):
        p = rkv.make_params(1, 1, g["T"], 1, 4, 32, 32, stride=g["s0"], alpha=alpha, n_sink=g["n_sink"])
        assert rkv.rkv_n_ref(p) == n


def test_dynamic_schedule_rejects_non_advancing_first_step(lib):
    # stride + floor(alpha (first - n_sink)) < 1 would not advance
    p = rkv.make_params(1, 1, 1000, 1, 4, 32, 32, stride=1, alpha=1.0, n_sink=10)
    assert rkv.rkv_n_ref(p) == -1
    a = ctypes.c_size_t()
    assert lib.rkv_query_sizes(ctypes.byref(p), ctypes.byref(a), None, None) == rkv.RKV_ERR_INVALID_ARG


def test_restore_validates_on_the_host(lib):
    pool = rkv.rkv_ref_pool(16, 16, 16, 16, 16)
    cache = rkv.rkv_cache(16, 16, 16)

    def call(p, Wd=16, sel=16, n_sel=4, base=10000.0, ok=16, ov=16, st=16):
        return lib.rkv_restore_kv(ctypes.byref(p), ctypes.byref(pool), ctypes.byref(cache), Wd, sel,
                                  n_sel, base, ok, ov, st, None)

    p = rkv.make_params(1, 1, 256, 8, 128, 1024, 512)
    assert call(p, n_sel=-1) == rkv.RKV_ERR_INVALID_ARG
    assert call(p, base=0.0) == rkv.RKV_ERR_INVALID_ARG
    assert call(p, base=float("inf")) == rkv.RKV_ERR_INVALID_ARG
    assert call(p, Wd=None) == rkv.RKV_ERR_INVALID_ARG
    assert call(p, ok=24) == rkv.RKV_ERR_ALIGNMENT
    assert call(p, n_sel=0) == rkv.RKV_OK                     # nothing to do, nothing launched
    assert call(rkv.make_params(1, 1, 256, 2, 64, 256, 64, kv_dtype="f32")) == rkv.RKV_ERR_UNSUPPORTED
    assert call(rkv.make_params(1, 1, 256, 8, 128, 1024, 384)) == rkv.RKV_ERR_UNSUPPORTED   # d_c
    assert call(rkv.make_params(1, 1, 256, 2, 48, 1024, 512)) == rkv.RKV_ERR_UNSUPPORTED    # D


def test_timeout_hook_validates_host_side(lib):
    # the timeout-path test hook checks its arguments on the host (no GPU needed)
    for cycles, skip in ((0, 0), (9999, 0), (3 * 10 ** 9, 0), (200000, -1)):
        assert lib.rkv_debug_wait_fault(cycles, skip) == rkv.RKV_ERR_INVALID_ARG


def test_guard_bytes_detect_a_write_past_the_end():
    # the test-support allocator behind the GPU tests' overrun checks, on host memory
    t, raw = rkv.guarded_empty((3, 5), torch.float32, "cpu", 64)
    t.fill_(1.0)
    assert rkv.guard_intact(t, raw)
    raw[t.numel() * t.element_size()] = 0          # the first byte past the tensor
    assert not rkv.guard_intact(t, raw)
    s, raw_s = rkv.guarded_empty((4,), torch.int32, "cpu", 16, fill=0)
    assert torch.equal(s, torch.zeros(4, dtype=torch.int32)) and rkv.guard_intact(s, raw_s)
    u, none = rkv.guarded_empty((2,), torch.uint8, "cpu", 0)
    assert none is None and rkv.guard_intact(u, none)
