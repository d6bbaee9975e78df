"""Host-side checks of the C ABI (no GPU): the library loads, exports every
declared entry point, computes layouts that match the oracle's specification,
and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import quantized_gemv_unpack_gb300 as q
from oracle import layout
from quantized_gemv_unpack_gb300 import build

from conftest import ROOT


@pytest.fixture(scope="module")
def L():
    build.build()
    return q.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "qmv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_constants_match_the_binding():
    src = open(os.path.join(ROOT, "include", "qmv.h")).read()
    defines = re.findall(r"^#define\s+(QMV_[A-Z0-9_]+)\s+([0-9u*()\s]+?)\s*(?:/\*.*)?$", src, flags=re.M)
    assert len(defines) >= 8
    for name, expr in defines:
        value = 1
        for factor in re.findall(r"[0-9]+", expr):   # a number or a product of numbers
            value *= int(factor)
        assert getattr(q, name) == value, name
    enums = re.findall(r"(QMV_[A-Z0-9_]+)\s*=\s*(-?[0-9]+)", src)
    assert len(enums) >= 10
    for name, value in enums:
        assert getattr(q, name) == int(value), name


def test_every_declared_symbol_is_exported(L):
    declared = _declared_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(L, name), f"{name} declared in qmv.h but not exported"
    assert sorted(q.EXPORTS) == declared


def test_desc_matches_oracle_layout(L):
    for fmt, sizes in [(q.QMV_TERNARY2, layout.ternary_sizes), (q.QMV_INT4, layout.int4_sizes)]:
        for N, K in [(1, 128), (7, 384), (4096, 4096), (1024, 5120), (5120, 25600)]:
            d = q.qmv_pack_desc(fmt, N, K)
            offs, total = layout.sections(sizes(N, K))
            assert [d.off[i] for i in range(2)] == offs
            assert [d.bytes[i] for i in range(2)] == sizes(N, K)
            assert d.total_bytes == total
            assert d.abi_version == q.QMV_ABI_VERSION and d.group == 128


def test_lut_desc_matches_oracle_layout(L):
    for N, K in [(1, 128), (31, 384), (33, 256), (4096, 4096), (1024, 5120), (5120, 25600)]:
        d = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, N, K)
        offs, total = layout.sections(layout.ternary_lut_sizes(N, K))
        assert [d.off[i] for i in range(2)] == offs
        assert [d.bytes[i] for i in range(2)] == layout.ternary_lut_sizes(N, K)
        assert d.total_bytes == total and d.format == q.QMV_TERNARY2_LUT


def test_lut_run_rejects_bad_arguments_on_the_host(L):
    d = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, 64, 256)
    rec = q.qmv_pack_desc(q.QMV_TERNARY2, 64, 256)
    # the lookup layout serves one activation row
    assert L.qmv_run_ternary(ctypes.byref(d), 256, 256, 2, 256, 256, 64, None) == q.QMV_ERR_UNSUPPORTED
    assert "M = 1" in q.qmv_last_error()
    assert L.qmv_run_ternary(ctypes.byref(d), 264, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ALIGN
    assert L.qmv_run_ternary(ctypes.byref(d), 256, None, 1, 256, 256, 64, None) == q.QMV_ERR_ARG
    bad = q.qmv_desc.from_buffer_copy(d)
    bad.bytes[1] -= 2
    assert L.qmv_run_ternary(ctypes.byref(bad), 256, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ARG
    # a record-layout desc in a lookup batch is rejected
    tasks = (q.qmv_task * 2)(q.qmv_task(ctypes.pointer(d), 256, 256, 256, 256, 64),
                             q.qmv_task(ctypes.pointer(rec), 256, 256, 256, 256, 64))
    assert L.qmv_run_batch(q.QMV_TERNARY2_LUT, tasks, 2, 1, None) == q.QMV_ERR_ARG
    assert "task 1" in q.qmv_last_error()


@pytest.mark.parametrize("args", [(q.QMV_TERNARY2, 0, 128), (q.QMV_TERNARY2, 4, 100), (q.QMV_INT4, 4, -128),
                                  (9, 4, 128), (q.QMV_TERNARY2_LUT, 4, 192), (q.QMV_TERNARY2_LUT, 4, 128, 64)])
def test_pack_desc_rejects_bad_shapes(L, args):
    with pytest.raises(q.QmvError) as e:
        q.qmv_pack_desc(*args)
    assert e.value.status == q.QMV_ERR_ARG


def test_cassandra_desc_needs_the_data(L):
    with pytest.raises(q.QmvError) as e:
        q.qmv_pack_desc(q.QMV_CASS, 4, 128)
    assert e.value.status == q.QMV_ERR_UNSUPPORTED


def test_run_rejects_bad_arguments_on_the_host(L):
    d = q.qmv_pack_desc(q.QMV_TERNARY2, 64, 256)
    # NULL desc, wrong format, misaligned pointers, short ldx and bad M are all found before any launch
    assert L.qmv_run_ternary(None, 256, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ARG
    assert L.qmv_run_int4(ctypes.byref(d), 256, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ARG
    assert L.qmv_run_ternary(ctypes.byref(d), 258, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ALIGN
    assert L.qmv_run_ternary(ctypes.byref(d), 256, 256, 1, 128, 256, 64, None) == q.QMV_ERR_ARG
    assert L.qmv_run_ternary(ctypes.byref(d), 256, 256, 1, 260, 256, 64, None) == q.QMV_ERR_ALIGN
    assert L.qmv_run_ternary(ctypes.byref(d), 256, 256, 0, 256, 256, 64, None) == q.QMV_ERR_ARG
    assert L.qmv_run_ternary(ctypes.byref(d), 256, 256, 17, 256, 256, 64, None) == q.QMV_ERR_ARG
    assert "M=17" in q.qmv_last_error()
    bad = q.qmv_desc.from_buffer_copy(d)
    bad.bytes[0] += 4
    assert L.qmv_run_ternary(ctypes.byref(bad), 256, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ARG
    bad = q.qmv_desc.from_buffer_copy(d)
    bad.abi_version = 99
    assert L.qmv_run_ternary(ctypes.byref(bad), 256, 256, 1, 256, 256, 64, None) == q.QMV_ERR_ARG
    assert L.qmv_run_batch(q.QMV_TERNARY2, None, 0, 1, None) == q.QMV_ERR_ARG
    both = q.qmv_pack_desc(q.QMV_TERNARY2, 64, 256)
    both.flags = q.QMV_FLAG_PATH_FMA | q.QMV_FLAG_PATH_MMA          # contradictory kernel choice
    assert L.qmv_run_ternary(ctypes.byref(both), 256, 256, 4, 256, 256, 64, None) == q.QMV_ERR_ARG


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(q, "_lib", None)
    monkeypatch.setattr(q, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        q.lib()


def test_batch_keeps_its_tensors_alive(L):
    """A prepared batch holds the tensors whose addresses it passes, so the caller's
    allocator cannot hand their memory out again while the batch may still launch."""
    import gc
    import weakref
    import torch
    d = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, 64, 256)
    w = torch.zeros(d.total_bytes, dtype=torch.uint8)
    x = torch.zeros((1, 256), dtype=torch.bfloat16)
    y = torch.zeros((1, 64), dtype=torch.float32)
    refs = [weakref.ref(t) for t in (w, x, y)]
    batch = q.Batch(q.QMV_TERNARY2_LUT, [(d, w, x, y)], 1)
    del w, x, y
    gc.collect()
    assert all(r() is not None for r in refs)
    del batch
    gc.collect()
    assert all(r() is None for r in refs)
