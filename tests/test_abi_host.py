"""The C-ABI library builds, loads and exports every declared entry point;
host-side argument checks answer without touching a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fastocr.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fastocr_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from conftest import build_library
    return ctypes.CDLL(build_library())


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ["fastocr_focal_attend", "fastocr_sparse_attend", "fastocr_rswa_attend",
                 "fastocr_full_attend", "fastocr_profiler_select", "fastocr_create"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    from dynamic_sparse_kv_gb300 import _native as N
    assert N.fastocr_abi_version() == 2
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert N.status_string(s) and N.status_string(s) != "unknown status"
    assert N.status_string(123) == "unknown status"


def test_host_checks_without_gpu(lib):
    from dynamic_sparse_kv_gb300 import _native as N
    L = N.lib
    h = ctypes.c_void_p()
    assert L.fastocr_create(None, ctypes.byref(h)) == N.FASTOCR_ERR_NULL
    bad = [
        N.fastocr_dims(0, 4, 2, 64, 1, 16, 8, 64, 2),      # batch 0
        N.fastocr_dims(1, 6, 4, 64, 1, 16, 8, 64, 2),      # H_q % H_kv
        N.fastocr_dims(1, 4, 2, 64, 7, 16, 8, 64, 2),      # dtype
        N.fastocr_dims(1, 4, 2, 64, 1, 12, 8, 64, 2),      # page size not a power of 2
        N.fastocr_dims(1, 4, 2, 64, 1, 16, 8, 64, 0),      # no layers
    ]
    for d in bad:
        assert L.fastocr_create(ctypes.byref(d), ctypes.byref(h)) == N.FASTOCR_ERR_INVALID
    unsupported = [
        N.fastocr_dims(1, 18, 2, 64, 1, 16, 8, 64, 2),     # group 9 > 8
        N.fastocr_dims(1, 4, 2, 96, 1, 16, 8, 64, 2),      # d = 96
        N.fastocr_dims(1, 4, 2, 64, 1, 16, 8, 20000, 2),   # too many image tokens
    ]
    for d in unsupported:
        assert L.fastocr_create(ctypes.byref(d), ctypes.byref(h)) == N.FASTOCR_ERR_UNSUPPORTED
    # NULL handle / pointers are refused before any CUDA call
    kv = N.fastocr_kv(None, None, None, None, 1)
    assert L.fastocr_full_attend(None, None, ctypes.byref(kv), None, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_sparse_attend(None, None, ctypes.byref(kv), None, None, 1, None, None,
                                   None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_sparse_attend_ex(None, None, ctypes.byref(kv), None, None, 1, None, None,
                                      N.SELECTION_FINAL, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_rswa_attend(None, None, ctypes.byref(kv), 0, 0, None, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_focal_attend(None, None, ctypes.byref(kv), None, 0.5, None, None, 1, None,
                                  -1, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_profiler_select(None, 1, None, None, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_profile_attend(None, None, ctypes.byref(kv), None, None, 0,
                                    None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_profiler_read(None, None, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_profiler_load(None, None, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_set_splits(None, 0, 1) == N.FASTOCR_ERR_NULL
    assert L.fastocr_set_variant(None, 0, 1) == N.FASTOCR_ERR_NULL
    assert L.fastocr_set_length_hint(None, 100) == N.FASTOCR_ERR_NULL
    assert L.fastocr_focal_scores(None, None, ctypes.byref(kv), None, None, None, 1,
                                  None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_select(None, ctypes.byref(kv), None, None, 1, 0.5, None, 1, None,
                            None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_destroy(None) == N.FASTOCR_OK
    # the read-only bandwidth probe checks its arguments before touching a GPU
    buf = (ctypes.c_uint8 * 64)()
    sink = ctypes.c_uint32()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    assert L.fastocr_read_probe(None, 32, ctypes.byref(sink), None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_read_probe(addr, 32, None, None) == N.FASTOCR_ERR_NULL
    for bad in (0, 8, 24, -16):
        assert L.fastocr_read_probe(addr, bad, ctypes.byref(sink), None) == N.FASTOCR_ERR_INVALID
    assert L.fastocr_read_probe(addr + 4, 32, ctypes.byref(sink), None) == N.FASTOCR_ERR_ALIGN
    # so does the SM copy: NULL, size, alignment and overlap before any CUDA call
    big = (ctypes.c_uint8 * 256)()
    a = (ctypes.addressof(big) + 15) // 16 * 16
    assert L.fastocr_copy(None, a, 32, None) == N.FASTOCR_ERR_NULL
    assert L.fastocr_copy(a, None, 32, None) == N.FASTOCR_ERR_NULL
    for bad in (8, 24, -16):
        assert L.fastocr_copy(a + 128, a, bad, None) == N.FASTOCR_ERR_INVALID
    assert L.fastocr_copy(a + 132, a, 32, None) == N.FASTOCR_ERR_ALIGN
    assert L.fastocr_copy(a + 128, a + 4, 32, None) == N.FASTOCR_ERR_ALIGN
    assert L.fastocr_copy(a + 16, a, 32, None) == N.FASTOCR_ERR_INVALID   # overlapping
    assert L.fastocr_copy(a, a + 16, 32, None) == N.FASTOCR_ERR_INVALID


def test_create_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from dynamic_sparse_kv_gb300 import _native as N
    d = N.fastocr_dims(1, 4, 2, 64, 1, 16, 8, 64, 2)
    h = ctypes.c_void_p()
    assert N.lib.fastocr_create(ctypes.byref(d), ctypes.byref(h)) == N.FASTOCR_ERR_NO_DEVICE


def test_header_compiles_as_c_and_cpp():
    import shutil
    import subprocess
    for comp, lang in (("gcc", "c"), ("g++", "c++")):
        if shutil.which(comp) is None:
            pytest.skip(f"{comp} not found")
        r = subprocess.run([comp, "-fsyntax-only", "-Wall", "-Werror", "-x", lang, HEADER],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_profile_schedule_windows(lib):
    """The decoder's profiling windows are the oracle's: one window without a
    period, a window of `window` steps at the start of every period with one."""
    import oracle.schedule as S
    from dynamic_sparse_kv_gb300 import ProfileSchedule
    for window, period in [(8, None), (0, None), (2, 7), (3, 4), (1, 2), (0, 5)]:
        sch = ProfileSchedule(window, period)
        got = [sch.position(t) for t in range(40)]
        assert got == [S.window_position(t, window, period) for t in range(40)]
    assert [ProfileSchedule(2, 7).position(t) for t in range(15)] == \
        [0, 1, -1, -1, -1, -1, -1, 0, 1, -1, -1, -1, -1, -1, 0]
    for bad in [(3, 3), (4, 2), (-1, None)]:
        with pytest.raises(ValueError):
            ProfileSchedule(*bad)


def test_host_io_output_chunks(lib):
    """A host-I/O captured step copies its outputs back in chunks of half the
    layers left: the chunks tile the layers in order, the last one is a
    single layer, and every chunk is at most as long as the layers after it
    plus one (so its copy has attention to hide behind)."""
    from dynamic_sparse_kv_gb300 import CapturedStep
    assert CapturedStep.output_chunks(28) == [13, 20, 23, 25, 26, 27]
    assert CapturedStep.output_chunks(1) == [0]
    for L in range(1, 70):
        ends = CapturedStep.output_chunks(L)
        assert ends[-1] == L - 1 and all(a < b for a, b in zip(ends, ends[1:]))
        starts = [0] + [e + 1 for e in ends[:-1]]
        assert ends[-1] - starts[-1] == 0
        for a, e in zip(starts, ends):
            assert (e - a + 1) <= (L - 1 - e) + 1
