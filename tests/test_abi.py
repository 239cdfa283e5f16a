"""Host-side checks of the C ABI: the library loads, exports what include/moda.h declares,
and rejects bad arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return binding.load_library()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moda_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("moda_fwd", "moda_bwd", "moda_bwd_workspace_bytes", "moda_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(binding.EXPORTS) <= set(declared_functions())


def test_status_strings_and_version(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert lib.moda_status_str(code).decode() == name
    assert lib.moda_version() >= 100


def desc(**kw):
    base = dict(B=1, H=4, Hkv=2, T=16, S=3, d=64, dtype=1, scale=0.0, slot_capacity=0)
    base.update(kw)
    return binding.moda_desc(base["B"], base["H"], base["Hkv"], base["T"], base["S"], base["d"], base["dtype"],
                             base["scale"], base["slot_capacity"])


FAKE = 1 << 20  # aligned fake device address: validation must fail before any use


def fwd(lib, d, ptrs=None):
    p = [ctypes.c_void_p(FAKE)] * 7 if ptrs is None else ptrs
    return lib.moda_fwd(ctypes.byref(d) if d is not None else None, *p, None)


@pytest.mark.parametrize("kw,status", [
    (dict(H=3, Hkv=2), 1), (dict(T=0), 1), (dict(B=0), 1), (dict(S=-1), 1), (dict(Hkv=0), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(dtype=7), 2), (dict(scale=float("nan")), 1),
    (dict(slot_capacity=-1), 1), (dict(S=4, slot_capacity=3), 1),
])
def test_forward_rejects_bad_desc(lib, kw, status):
    assert fwd(lib, desc(**kw)) == status


def test_forward_rejects_null_and_misaligned(lib):
    assert fwd(lib, None) == 1
    ptrs = [ctypes.c_void_p(FAKE)] * 7
    for i in (0, 1, 2, 5):
        bad = list(ptrs)
        bad[i] = None
        assert fwd(lib, desc(), bad) == 1
    for i in range(7):
        bad = list(ptrs)
        bad[i] = ctypes.c_void_p(FAKE + 8)
        assert fwd(lib, desc(), bad) == 1
    # depth pointers may be null only when S == 0
    bad = list(ptrs)
    bad[3] = None
    assert fwd(lib, desc(S=3), bad) == 1


def test_backward_workspace_contract(lib):
    d = desc(B=2, H=4, Hkv=2, T=100, S=3, d=64)
    need = lib.moda_bwd_workspace_bytes(ctypes.byref(d))
    assert need >= 2 * 4 * 100 * 4 + 2 * 4 * 100 * 64 * 4
    assert lib.moda_bwd_workspace_bytes(ctypes.byref(desc(H=3))) == 0
    ptrs = [ctypes.c_void_p(FAKE)] * 13
    ws = ctypes.c_void_p(FAKE)
    # too small / missing workspace
    assert lib.moda_bwd(ctypes.byref(d), *ptrs, ws, ctypes.c_size_t(need - 1), None) == 5
    assert lib.moda_bwd(ctypes.byref(d), *ptrs, None, ctypes.c_size_t(need), None) == 5
    # workspace not 256-byte aligned
    assert lib.moda_bwd(ctypes.byref(d), *ptrs, ctypes.c_void_p(FAKE + 16), ctypes.c_size_t(need), None) == 1


def test_depth_writes_reject_bad_arguments(lib):
    """Slot out of range (of the slots in memory), fp32, null or misaligned pointers,
    d_model not a multiple of 8: all refused before any launch."""
    f = ctypes.c_void_p(FAKE)
    store = lambda d, slot, ptrs=None: lib.moda_depth_store_kv(ctypes.byref(d), slot, *(ptrs or [f] * 4), None)  # noqa: E731
    assert store(desc(S=3), -1) == 1
    assert store(desc(S=3), 3) == 1
    assert store(desc(S=3, slot_capacity=8), 8) == 1
    assert store(desc(S=0), 0) == 1
    assert store(desc(S=3, dtype=0), 0) == 2
    for i in range(4):
        bad = [f] * 4
        bad[i] = None
        assert store(desc(), 0, bad) == 1
        bad[i] = ctypes.c_void_p(FAKE + 4)
        assert store(desc(), 0, bad) == 1
    project = lambda d, slot, dm, ptrs=None: lib.moda_depth_project_kv(  # noqa: E731
        ctypes.byref(d), slot, dm, *(ptrs or [f] * 5), None)
    assert project(desc(S=3), 3, 64) == 1
    assert project(desc(S=3), 0, 12) == 1
    assert project(desc(S=3), 0, 0) == 1
    assert project(desc(S=3, dtype=0), 0, 64) == 2
    for i in range(5):
        bad = [f] * 5
        bad[i] = ctypes.c_void_p(FAKE + 8)
        assert project(desc(), 0, 64, bad) == 1


def test_decode_rejects_bad_arguments(lib):
    """Cache capacity below T, fp32, null pointers: refused before any launch."""
    f = ctypes.c_void_p(FAKE)
    dec = lambda d, cap, ptrs=None: lib.moda_decode(  # noqa: E731
        ctypes.byref(d), ctypes.c_int64(cap), *(ptrs or [f] * 6), None, f, ctypes.c_size_t(1 << 20), None)
    assert dec(desc(T=16), 15) == 1
    assert dec(desc(dtype=0), 0) == 2
    bad = [f] * 6  # q, k_cache, v_cache, kd, vd, o
    bad[0] = None
    assert dec(desc(), 0, bad) == 1
    bad = [f] * 6
    bad[3] = None  # depth keys missing while S > 0
    assert dec(desc(S=3), 0, bad) == 1


def test_context_parallel_calls_reject_bad_arguments(lib):
    """Chunk geometry (delta < 0, Tk < 1, Tk > T + delta), a missing lse, null or
    misaligned pointers: refused before any launch.  T = 16 query positions."""
    f = ctypes.c_void_p(FAKE)
    d = desc()
    # pointers: q, k, v, kd, vd, o, lse
    fp = lambda Tk, delta, ptrs=None: lib.moda_fwd_partial(  # noqa: E731
        ctypes.byref(d), Tk, delta, *(ptrs or [f] * 7), None)
    assert fp(16, -1) == 1
    assert fp(0, 0) == 1
    assert fp(17, 0) == 1        # key 16 is seen by no query
    assert fp(40, 23) == 1       # T + delta = 39 < 40
    assert fp(16, 0, [f] * 6 + [None]) == 1  # lse required
    for i in range(7):
        bad = [f] * 7
        bad[i] = ctypes.c_void_p(FAKE + 8)
        assert fp(16, 0, bad) == 1
    ws = ctypes.c_void_p(FAKE)
    need = ctypes.c_size_t(lib.moda_bwd_workspace_bytes(ctypes.byref(d)))
    bp = lambda Tk, delta, ptrs=None: lib.moda_bwd_partial(  # noqa: E731
        ctypes.byref(d), Tk, delta, *(ptrs or [f] * 13), ws, need, None)
    assert bp(16, -1) == 1
    assert bp(17, 0) == 1
    assert bp(16, 0, [f] * 9 + [None] + [f] * 3) == 1  # dk accumulator missing
    assert lib.moda_bwd_partial(ctypes.byref(d), 16, 0, *([f] * 13), ws, ctypes.c_size_t(need.value - 1),
                                None) == 5
    mp = lambda ptrs, dd=d: lib.moda_merge_partial(ctypes.byref(dd), *ptrs[:4], 0, ptrs[4], None)  # noqa: E731
    for i in range(4):
        bad = [f] * 5
        bad[i] = None
        assert mp(bad) == 1
    for i in range(5):
        bad = [f] * 5
        bad[i] = ctypes.c_void_p(FAKE + 4)
        assert mp(bad) == 1
    assert mp([f] * 5, desc(d=96)) == 2
    cv = lib.moda_convert_f32
    assert cv(ctypes.c_int64(-1), f, 1, f, None) == 1
    assert cv(ctypes.c_int64(16), f, 7, f, None) == 2
    assert cv(ctypes.c_int64(16), ctypes.c_void_p(FAKE + 4), 1, f, None) == 1
    assert cv(ctypes.c_int64(0), None, 1, None, None) == 0  # nothing to do, nothing launched
