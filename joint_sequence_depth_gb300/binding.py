"""Python binding of the MoDA C ABI (include/moda.h): argument marshalling only.

Each function takes torch CUDA tensors, allocates missing outputs with torch
(device memory is torch's), and hands raw pointers to ``libmoda.so``.  Every
step of the computation runs in the library's CUDA kernels; if the library is
missing this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

MODA_OK = 0
STATUS_NAMES = {0: "MODA_OK", 1: "MODA_ERR_INVALID_ARG", 2: "MODA_ERR_UNSUPPORTED", 3: "MODA_ERR_CUDA",
                4: "MODA_ERR_TIMEOUT", 5: "MODA_ERR_WORKSPACE"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}

# Names of every function include/moda.h declares.
EXPORTS = ("moda_fwd", "moda_bwd", "moda_bwd_workspace_bytes", "moda_device_status",
           "moda_status_str",
           "moda_version", "moda_launch_count", "moda_bwd_noalloc", "moda_bwd_noalloc_max_workspace_bytes",
           "moda_bwd_profiled", "moda_selftest_wait_timeout", "moda_decode", "moda_decode_workspace_bytes",
           "moda_depth_store_kv", "moda_depth_project_kv", "moda_fwd_partial", "moda_merge_partial",
           "moda_bwd_partial", "moda_convert_f32")


class MODAError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class moda_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("T", ctypes.c_int32),
                ("S", ctypes.c_int32), ("d", ctypes.c_int32), ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("slot_capacity", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def load_library():
    """Loads libmoda.so (built in-tree by ``build.build()``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libmoda.so is not built ({_build.LIB}); run __graft_entry__.build()")
            lib = ctypes.CDLL(_build.LIB)
            p, d = ctypes.c_void_p, ctypes.POINTER(moda_desc)
            lib.moda_fwd.argtypes = [d, p, p, p, p, p, p, p, p]
            lib.moda_fwd.restype = ctypes.c_int
            lib.moda_bwd_workspace_bytes.argtypes = [d]
            lib.moda_bwd_workspace_bytes.restype = ctypes.c_size_t
            lib.moda_bwd.argtypes = [d] + [p] * 14 + [ctypes.c_size_t, p]
            lib.moda_bwd.restype = ctypes.c_int
            lib.moda_bwd_profiled.argtypes = [d] + [p] * 14 + [ctypes.c_size_t, p, ctypes.POINTER(p), ctypes.c_int32]
            lib.moda_bwd_profiled.restype = ctypes.c_int
            lib.moda_device_status.argtypes = [ctypes.c_int, p]
            lib.moda_device_status.restype = ctypes.c_int
            lib.moda_status_str.argtypes = [ctypes.c_int]
            lib.moda_status_str.restype = ctypes.c_char_p
            lib.moda_version.argtypes = []
            lib.moda_version.restype = ctypes.c_int32
            lib.moda_launch_count.argtypes = []
            lib.moda_launch_count.restype = ctypes.c_int64
            lib.moda_bwd_noalloc.argtypes = [d] + [p] * 14
            lib.moda_bwd_noalloc.restype = ctypes.c_int
            lib.moda_bwd_noalloc_max_workspace_bytes.argtypes = []
            lib.moda_bwd_noalloc_max_workspace_bytes.restype = ctypes.c_size_t
            lib.moda_selftest_wait_timeout.argtypes = [ctypes.c_uint64, p]
            lib.moda_selftest_wait_timeout.restype = ctypes.c_int
            lib.moda_decode_workspace_bytes.argtypes = [d]
            lib.moda_decode_workspace_bytes.restype = ctypes.c_size_t
            lib.moda_decode.argtypes = [d, ctypes.c_int64] + [p] * 8 + [ctypes.c_size_t, p]
            lib.moda_depth_store_kv.argtypes = [d, ctypes.c_int32] + [p] * 5
            lib.moda_depth_store_kv.restype = ctypes.c_int
            lib.moda_depth_project_kv.argtypes = [d, ctypes.c_int32, ctypes.c_int32] + [p] * 6
            lib.moda_depth_project_kv.restype = ctypes.c_int
            lib.moda_decode.restype = ctypes.c_int
            i32 = ctypes.c_int32
            lib.moda_fwd_partial.argtypes = [d, i32, i32] + [p] * 8
            lib.moda_fwd_partial.restype = ctypes.c_int
            lib.moda_merge_partial.argtypes = [d, p, p, p, p, i32, p, p]
            lib.moda_merge_partial.restype = ctypes.c_int
            lib.moda_bwd_partial.argtypes = [d, i32, i32] + [p] * 14 + [ctypes.c_size_t, p]
            lib.moda_bwd_partial.restype = ctypes.c_int
            lib.moda_convert_f32.argtypes = [ctypes.c_int64, p, i32, p, p]
            lib.moda_convert_f32.restype = ctypes.c_int
            _lib = lib
    return _lib


def make_desc(B, H, Hkv, T, S, d, dtype, scale=None, slot_capacity=0) -> moda_desc:
    return moda_desc(B, H, Hkv, T, S, d, DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype),
                     float(scale or 0.0), int(slot_capacity))


def _slots(kd, slots):
    """(S read, slot capacity) for a depth tensor whose dim 3 holds the slots in memory:
    ``slots=None`` reads them all."""
    if kd is None:
        return 0, 0
    cap = kd.shape[3]
    if slots is None or int(slots) == cap:
        return cap, 0
    return int(slots), cap


def _desc_from(q, k, kd, scale, slots=None):
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    S, cap = _slots(kd, slots)
    if q.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    return make_desc(B, H, Hkv, T, S, d, q.dtype, scale, cap)


def _mem_slots(desc):
    return desc.slot_capacity if desc.slot_capacity > 0 else desc.S


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _check_like(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def moda_fwd(q, k, v, kd, vd, o=None, lse=None, scale=None, stream=None, slots=None):
    """Joint sequence/depth attention forward.  Returns (o [B,H,T,d], lse [B,H,T] float32).
    ``slots``: read only slots 0..slots-1 of kd/vd[B,Hkv,T,C,d] (a bounded slot buffer of
    capacity C, see slot_capacity in include/moda.h); None reads all C."""
    desc = _desc_from(q, k, kd, scale, slots)
    B, H, T, d = q.shape
    for t, name in ((k, "k"), (v, "v")):
        _check_like(t, q.dtype, (B, desc.Hkv, T, d), name)
    if desc.S:
        for t, name in ((kd, "kd"), (vd, "vd")):
            _check_like(t, q.dtype, (B, desc.Hkv, T, _mem_slots(desc), d), name)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    st = load_library().moda_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(kd) if desc.S else None,
                                 _ptr(vd) if desc.S else None, _ptr(o), _ptr(lse), _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_fwd")
    return o, lse


def moda_bwd_workspace_bytes(desc: moda_desc) -> int:
    return int(load_library().moda_bwd_workspace_bytes(ctypes.byref(desc)))


def moda_bwd(q, k, v, kd, vd, o, lse, dout, grads=None, workspace=None, scale=None, stream=None, events=None,
             slots=None):
    """Backward of moda_fwd.  Returns (dq, dk, dv, dkd, dvd) in the input dtype.  ``events``
    (optional list of torch.cuda.Event) are recorded after each internal stage, see
    moda_bwd_profiled in include/moda.h.  ``slots`` as for moda_fwd (dkd/dvd of the
    unread slots come back as zero)."""
    desc = _desc_from(q, k, kd, scale, slots)
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty_like(kd) if desc.S else None, torch.empty_like(vd) if desc.S else None)
    dq, dk, dv, dkd, dvd = grads
    need = moda_bwd_workspace_bytes(desc)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    args = (ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(kd) if desc.S else None,
            _ptr(vd) if desc.S else None, _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(dkd) if desc.S else None, _ptr(dvd) if desc.S else None, _ptr(workspace),
            ctypes.c_size_t(workspace.numel()), _stream(stream))
    if events is None:
        st = load_library().moda_bwd(*args)
    else:
        handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        st = load_library().moda_bwd_profiled(*args, handles, len(events))
    if st != MODA_OK:
        raise MODAError(st, "moda_bwd")
    return dq, dk, dv, dkd, dvd


def moda_device_status(clear=True, stream=None) -> int:
    return int(load_library().moda_device_status(1 if clear else 0, _stream(stream)))


def moda_selftest_wait_timeout(limit_ns=20_000_000, stream=None) -> int:
    """Runs the bounded-wait self-test kernel on the current device; returns the status
    it produced (MODA_ERR_TIMEOUT = 4 when the failure path worked)."""
    return int(load_library().moda_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def moda_launch_count() -> int:
    """Kernels the library has launched since it was loaded."""
    return int(load_library().moda_launch_count())


def moda_bwd_noalloc(q, k, v, kd, vd, o, lse, dout, grads, scale=None, stream=None, slots=None):
    """moda_bwd without a workspace argument, for callers that cannot allocate device memory:
    the library uses its own fixed device array (see include/moda.h).  ``grads`` must be
    preallocated (dq, dk, dv, dkd, dvd); returns them."""
    desc = _desc_from(q, k, kd, scale, slots)
    dq, dk, dv, dkd, dvd = grads
    st = load_library().moda_bwd_noalloc(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(kd) if desc.S else None, _ptr(vd) if desc.S else None,
        _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dkd) if desc.S else None,
        _ptr(dvd) if desc.S else None, _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_bwd_noalloc")
    return grads


def moda_bwd_noalloc_max_workspace_bytes() -> int:
    return int(load_library().moda_bwd_noalloc_max_workspace_bytes())


def moda_decode_workspace_bytes(desc: moda_desc) -> int:
    return int(load_library().moda_decode_workspace_bytes(ctypes.byref(desc)))


def moda_decode(q, k_cache, v_cache, kd, vd, T=None, o=None, lse=None, workspace=None, scale=None, stream=None,
                slots=None):
    """Decode step (moda_decode in include/moda.h): q[B,H,d] of the newest position,
    k_cache/v_cache[B,Hkv,capacity,d] holding positions 0..T-1 (T defaults to the
    capacity), kd/vd[B,Hkv,C,d] (the newest position's depth slots, None when there are
    none; only slots 0..slots-1 are read when ``slots`` is given).
    Returns (o[B,H,d], lse[B,H] float32)."""
    B, H, d = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    S, slot_cap = (0, 0) if kd is None else _slots(kd.unsqueeze(2), slots)
    T = cap if T is None else int(T)
    desc = make_desc(B, H, Hkv, T, S, d, q.dtype, scale, slot_cap)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    need = moda_decode_workspace_bytes(desc)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = load_library().moda_decode(ctypes.byref(desc), ctypes.c_int64(cap), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(kd) if S else None, _ptr(vd) if S else None, _ptr(o), _ptr(lse),
                                    _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_decode")
    return o, lse


def moda_depth_store_kv(k, v, kd, vd, slot, stream=None):
    """Writes k, v [B,Hkv,T,d] into slot ``slot`` of kd, vd [B,Hkv,T,S,d] in place
    (moda_depth_store_kv in include/moda.h); returns (kd, vd)."""
    B, Hkv, T, S, d = kd.shape
    desc = make_desc(B, Hkv, Hkv, T, S, d, k.dtype, None)
    st = load_library().moda_depth_store_kv(ctypes.byref(desc), int(slot), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd),
                                            _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_depth_store_kv")
    return kd, vd


def moda_depth_project_kv(x, wk, wv, kd, vd, slot, stream=None):
    """Writes x[B,T,Dm] @ wk and x @ wv (wk, wv [Dm, Hkv*d]) into slot ``slot`` of kd, vd
    [B,Hkv,T,S,d] in place (moda_depth_project_kv in include/moda.h); returns (kd, vd)."""
    B, Hkv, T, S, d = kd.shape
    Dm = x.shape[2]
    desc = make_desc(B, Hkv, Hkv, T, S, d, x.dtype, None)
    st = load_library().moda_depth_project_kv(ctypes.byref(desc), int(slot), int(Dm), _ptr(x), _ptr(wk), _ptr(wv),
                                              _ptr(kd), _ptr(vd), _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_depth_project_kv")
    return kd, vd


# ---------------------------------------------------------------- context parallelism
def _chunk_desc(q, k, kd, scale, slots):
    """Description of a (query chunk, key chunk) pair: T from q, Tk from k."""
    desc = _desc_from(q, k, kd, scale, slots)
    B, H, T, d = q.shape
    if k.shape[0] != B or k.shape[3] != d or k.dtype != q.dtype:
        raise ValueError("k: batch, head dim and dtype must match q")
    return desc, int(k.shape[2])


def moda_fwd_partial(q, k, v, kd, vd, delta, o=None, lse=None, scale=None, stream=None, slots=None):
    """Partial forward of a query chunk q[B,H,T,d] against a key chunk k, v[B,Hkv,Tk,d]
    (moda_fwd_partial in include/moda.h): key j visible to query t iff j <= t + delta;
    kd/vd (the query chunk's own depth slots) or None.  Returns (o, lse) over this chunk's
    keys alone."""
    desc, Tk = _chunk_desc(q, k, kd, scale, slots)
    B, H, T, d = q.shape
    _check_like(v, q.dtype, k.shape, "v")
    if desc.S:
        for t, name in ((kd, "kd"), (vd, "vd")):
            _check_like(t, q.dtype, (B, desc.Hkv, T, _mem_slots(desc), d), name)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    st = load_library().moda_fwd_partial(ctypes.byref(desc), int(Tk), int(delta), _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(kd) if desc.S else None, _ptr(vd) if desc.S else None, _ptr(o),
                                         _ptr(lse), _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_fwd_partial")
    return o, lse


def moda_merge_partial(o_acc, lse_acc, o_part, lse_part, first=False, o_out=None, stream=None):
    """Merges a partial state (o_part [B,H,T,d], lse_part [B,H,T]) into the float32 running
    state (o_acc, lse_acc) in place (moda_merge_partial in include/moda.h); ``o_out``
    (o_part's dtype) optionally receives the merged O.  Returns (o_acc, lse_acc)."""
    B, H, T, d = o_part.shape
    _check_like(o_acc, torch.float32, o_part.shape, "o_acc")
    _check_like(lse_acc, torch.float32, (B, H, T), "lse_acc")
    _check_like(lse_part, torch.float32, (B, H, T), "lse_part")
    if o_out is not None:
        _check_like(o_out, o_part.dtype, o_part.shape, "o_out")
    desc = make_desc(B, H, H, T, 0, d, o_part.dtype, None)
    st = load_library().moda_merge_partial(ctypes.byref(desc), _ptr(o_acc), _ptr(lse_acc), _ptr(o_part),
                                           _ptr(lse_part), 1 if first else 0, _ptr(o_out), _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_merge_partial")
    return o_acc, lse_acc


def moda_bwd_partial(q, k, v, kd, vd, o, lse, dout, delta, dq_acc, dk_acc, dv_acc, dkd=None, dvd=None,
                     workspace=None, scale=None, stream=None, slots=None):
    """Adds one (query chunk, key chunk) pair's gradients to the float32 accumulators
    dq_acc [B,H,T,d], dk_acc/dv_acc [B,Hkv,Tk,d] (moda_bwd_partial in include/moda.h); o,
    lse are the query chunk's merged output and lse.  With depth slots (kd, vd not None)
    dkd, dvd are written.  Returns (dq_acc, dk_acc, dv_acc, dkd, dvd)."""
    desc, Tk = _chunk_desc(q, k, kd, scale, slots)
    _check_like(dq_acc, torch.float32, q.shape, "dq_acc")
    _check_like(dk_acc, torch.float32, k.shape, "dk_acc")
    _check_like(dv_acc, torch.float32, k.shape, "dv_acc")
    if desc.S:
        if dkd is None:
            dkd = torch.empty_like(kd)
        if dvd is None:
            dvd = torch.empty_like(vd)
    need = moda_bwd_workspace_bytes(desc)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = load_library().moda_bwd_partial(
        ctypes.byref(desc), int(Tk), int(delta), _ptr(q), _ptr(k), _ptr(v), _ptr(kd) if desc.S else None,
        _ptr(vd) if desc.S else None, _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc),
        _ptr(dkd) if desc.S else None, _ptr(dvd) if desc.S else None, _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_bwd_partial")
    return dq_acc, dk_acc, dv_acc, dkd, dvd


def moda_convert_f32(src, dtype, out=None, stream=None):
    """Rounds a float32 tensor to ``dtype`` (torch.bfloat16 or torch.float32) in the library's
    kernel (moda_convert_f32 in include/moda.h)."""
    if src.dtype != torch.float32:
        raise ValueError("src must be float32")
    if out is None:
        out = torch.empty(src.shape, dtype=dtype, device=src.device)
    _check_like(out, dtype, src.shape, "out")
    st = load_library().moda_convert_f32(ctypes.c_int64(src.numel()), _ptr(src), DTYPES[dtype], _ptr(out),
                                         _stream(stream))
    if st != MODA_OK:
        raise MODAError(st, "moda_convert_f32")
    return out
