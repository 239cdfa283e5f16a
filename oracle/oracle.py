"""ctypes front end of the float64 MoDA oracle (``moda_oracle.cpp``).

TEST INFRASTRUCTURE ONLY.  What each call computes is stated in the C++ file's
header; this module only compiles it with gcc (no CUDA) and marshals numpy
arrays.  Inputs are numpy arrays in one storage type for all operands:
float64, float32, or bfloat16 carried as uint16 bit patterns (the upper half of
a float32).  Every output is float64.

Definition followed: "Mixture-of-Depths Attention", frame "One denominator
allocates probability across both memories" (Sec. 2.2, Algorithm 1), with the
masks of frame "Backup: grouped indexing preserves the correct token map".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moda_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoda_oracle.so")

DTYPE_F64, DTYPE_F32, DTYPE_BF16 = 0, 1, 2

_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("Hkv", ctypes.c_int64),
        ("T", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("d", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("seq_window", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("nthreads", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) into oracle/_build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            dp = ctypes.POINTER(_Dims)
            lib.orc_cores.restype = ctypes.c_int
            lib.orc_forward.argtypes = [dp, p, p, p, p, p, p, ctypes.c_int64, p, p]
            lib.orc_forward.restype = ctypes.c_int
            lib.orc_backward_positions.argtypes = [dp, p, p, p, p, p, p, p, ctypes.c_int64, p, p, p]
            lib.orc_backward_positions.restype = ctypes.c_int
            lib.orc_backward_keys.argtypes = [dp, p, p, p, p, p, p, p, ctypes.c_int64, p, p]
            lib.orc_backward_keys.restype = ctypes.c_int
            _lib = lib
    return _lib


def cores() -> int:
    """Host cores in this process's affinity mask (the oracle's default thread count)."""
    return int(_load().orc_cores())


def _storage(arrs):
    dt = arrs[0].dtype
    for a in arrs:
        if a.dtype != dt:
            raise TypeError("all oracle inputs must share one storage type")
    if dt == np.float64:
        return DTYPE_F64
    if dt == np.float32:
        return DTYPE_F32
    if dt == np.uint16:
        return DTYPE_BF16
    raise TypeError(f"unsupported oracle storage type {dt}")


def _dims(q, k, kd, scale, seq_window, nthreads, dtype):
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    S = kd.shape[3]
    if k.shape != (B, Hkv, T, d) or kd.shape != (B, Hkv, T, S, d):
        raise ValueError("shape mismatch: q[B,H,T,d], k/v[B,Hkv,T,d], kd/vd[B,Hkv,T,S,d]")
    if H % Hkv:
        raise ValueError("H must be a multiple of Hkv")
    return _Dims(B, H, Hkv, T, S, d, float(scale or 0.0), int(seq_window), dtype, int(nthreads))


def _c(a):
    return np.ascontiguousarray(a)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def forward(q, k, v, kd, vd, scale=None, rows=None, seq_window=0, nthreads=0):
    """Joint sequence/depth softmax attention.

    q[B,H,T,d], k/v[B,Hkv,T,d], kd/vd[B,Hkv,T,S,d] -> (o, lse).
    rows=None: o[B,H,T,d], lse[B,H,T].  rows = flat indices (b*H+h)*T+t:
    o[n,d], lse[n].  seq_window=w>0 keeps only sequence keys t-w < j <= t
    (w=1: the softmax over {t} and the depth slots).
    """
    q, k, v, kd, vd = map(_c, (q, k, v, kd, vd))
    D = _dims(q, k, kd, scale, seq_window, nthreads, _storage([q, k, v, kd, vd]))
    if rows is None:
        o = np.empty(q.shape, np.float64)
        lse = np.empty(q.shape[:3], np.float64)
        rp, n = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.size
        o = np.empty((n, q.shape[3]), np.float64)
        lse = np.empty((n,), np.float64)
        rp = _ptr(rows)
    rc = _load().orc_forward(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd), rp, n,
                             _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle rejected the dimensions")
    return o, lse


def backward_positions(q, k, v, kd, vd, dout, positions=None, scale=None, seq_window=0, nthreads=0):
    """Position part of the backward: for flat positions p=(b*Hkv+g)*T+t (all when None),
    returns dq[n,G,d] (the G heads of the position), dkd[n,S,d], dvd[n,S,d]."""
    q, k, v, kd, vd, dout = map(_c, (q, k, v, kd, vd, dout))
    D = _dims(q, k, kd, scale, seq_window, nthreads, _storage([q, k, v, kd, vd, dout]))
    G = D.H // D.Hkv
    if positions is None:
        n, pp = D.B * D.Hkv * D.T, None
    else:
        positions = np.ascontiguousarray(positions, dtype=np.int64)
        n, pp = positions.size, _ptr(positions)
    dq = np.empty((n, G, D.d), np.float64)
    dkd = np.empty((n, D.S, D.d), np.float64)
    dvd = np.empty((n, D.S, D.d), np.float64)
    rc = _load().orc_backward_positions(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd),
                                        _ptr(dout), pp, n if pp is not None else 0, _ptr(dq), _ptr(dkd),
                                        _ptr(dvd))
    if rc:
        raise ValueError("oracle rejected the dimensions")
    return dq, dkd, dvd


def backward_keys(q, k, v, kd, vd, dout, keys=None, scale=None, seq_window=0, nthreads=0):
    """Key-column part of the backward: for flat keys p=(b*Hkv+g)*T+j (all when None),
    returns dk[n,d], dv[n,d] summed over the G heads and every row t >= j."""
    q, k, v, kd, vd, dout = map(_c, (q, k, v, kd, vd, dout))
    D = _dims(q, k, kd, scale, seq_window, nthreads, _storage([q, k, v, kd, vd, dout]))
    if keys is None:
        n, kp = D.B * D.Hkv * D.T, None
    else:
        keys = np.ascontiguousarray(keys, dtype=np.int64)
        n, kp = keys.size, _ptr(keys)
    dk = np.empty((n, D.d), np.float64)
    dv = np.empty((n, D.d), np.float64)
    rc = _load().orc_backward_keys(ctypes.byref(D), _ptr(q), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd),
                                   _ptr(dout), kp, n if kp is not None else 0, _ptr(dk), _ptr(dv))
    if rc:
        raise ValueError("oracle rejected the dimensions")
    return dk, dv


def backward(q, k, v, kd, vd, dout, scale=None, seq_window=0, nthreads=0):
    """Full backward: (dq[B,H,T,d], dk[B,Hkv,T,d], dv, dkd[B,Hkv,T,S,d], dvd), float64."""
    B, H, T, d = q.shape
    Hkv, S = k.shape[1], kd.shape[3]
    G = H // Hkv
    dqp, dkd, dvd = backward_positions(q, k, v, kd, vd, dout, None, scale, seq_window, nthreads)
    dk, dv = backward_keys(q, k, v, kd, vd, dout, None, scale, seq_window, nthreads)
    # positions are ordered (b, g, t); dq rows of a position are heads g*G .. g*G+G-1
    dq = dqp.reshape(B, Hkv, T, G, d).transpose(0, 1, 3, 2, 4).reshape(B, H, T, d)
    return (dq, dk.reshape(B, Hkv, T, d), dv.reshape(B, Hkv, T, d),
            dkd.reshape(B, Hkv, T, S, d), dvd.reshape(B, Hkv, T, S, d))


def _widen(a):
    """Stored values as float64: float64 as is, float32 widened, bf16 (uint16 bit patterns,
    the upper half of a float32) widened exactly."""
    a = np.asarray(a)
    if a.dtype == np.float64:
        return a
    if a.dtype == np.float32:
        return a.astype(np.float64)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unsupported storage type {a.dtype}")


def decode(q, k, v, kd, vd, scale=None):
    """One decode step of the joint operator ("Mixture-of-Depths Attention", frame "One
    denominator allocates probability across both memories", with the decode cache of the
    Table 1 frame "Depth compute still accumulates quadratically in depth"): the query of
    the newest position T-1 attends to every cached sequence key j <= T-1 and to the S depth
    slots of its own position, under one softmax.

    q[B,H,d], k/v[B,Hkv,T,d] (the sequence cache, newest position included),
    kd/vd[B,Hkv,S,d] (the depth slots of the newest position) -> (o[B,H,d], lse[B,H]),
    float64.  Plain definition: gather the scores, subtract the maximum, sum, divide once.
    """
    Q, K, V, KD, VD = (_widen(a) for a in (q, k, v, kd, vd))
    B, H, d = Q.shape
    Hkv, T = K.shape[1], K.shape[2]
    S = KD.shape[2]
    if K.shape != (B, Hkv, T, d) or V.shape != K.shape or KD.shape != (B, Hkv, S, d) or VD.shape != KD.shape:
        raise ValueError("shape mismatch: q[B,H,d], k/v[B,Hkv,T,d], kd/vd[B,Hkv,S,d]")
    if H % Hkv or T < 1:
        raise ValueError("H must be a multiple of Hkv and T >= 1")
    G = H // Hkv
    sc = float(scale) if scale else 1.0 / np.sqrt(d)
    o = np.empty((B, H, d), np.float64)
    lse = np.empty((B, H), np.float64)
    for b in range(B):
        for h in range(H):
            g = h // G
            scores = np.concatenate([K[b, g] @ Q[b, h], KD[b, g] @ Q[b, h]]) * sc
            m = scores.max()
            e = np.exp(scores - m)
            z = e.sum()
            o[b, h] = (e[:T] @ V[b, g] + e[T:] @ VD[b, g]) / z
            lse[b, h] = m + np.log(z)
    return o, lse


def depth_store(k, v, kd, vd, slot):
    """Reuse of the attention KV as a depth slot ("Mixture-of-Depths Attention", frame
    "Reuse attention KV; add a projection for FFN inputs", step 3): the layer's k, v
    [B,Hkv,T,d] become slot `slot` of kd, vd [B,Hkv,T,S,d]; every other slot is kept.
    Returns new float64 arrays."""
    K, V, KD, VD = (_widen(a).copy() for a in (k, v, kd, vd))
    if K.shape != KD.shape[:3] + KD.shape[4:] or V.shape != K.shape or VD.shape != KD.shape:
        raise ValueError("shape mismatch: k/v[B,Hkv,T,d], kd/vd[B,Hkv,T,S,d]")
    if not 0 <= slot < KD.shape[3]:
        raise ValueError("slot out of range")
    KD[:, :, :, slot, :] = K
    VD[:, :, :, slot, :] = V
    return KD, VD


def depth_project(x, wk, wv, kd, vd, slot):
    """The FFN input projected into an additional depth slot (same frame, step 4):
    kd[b,g,t,slot,c] = sum_m x[b,t,m] wk[m, g*d + c] and vd likewise with wv, for
    x[B,T,Dm], wk/wv[Dm, Hkv*d], kd/vd[B,Hkv,T,S,d]; every other slot is kept.
    A plain float64 matmul per (b); returns new float64 arrays."""
    X, WK, WV, KD, VD = (_widen(a) for a in (x, wk, wv, kd, vd))
    KD, VD = KD.copy(), VD.copy()
    B, T, Dm = X.shape
    Hkv, S, d = KD.shape[1], KD.shape[3], KD.shape[4]
    if KD.shape[:3] != (B, Hkv, T) or WK.shape != (Dm, Hkv * d) or WV.shape != WK.shape or VD.shape != KD.shape:
        raise ValueError("shape mismatch: x[B,T,Dm], wk/wv[Dm,Hkv*d], kd/vd[B,Hkv,T,S,d]")
    if not 0 <= slot < S:
        raise ValueError("slot out of range")
    for b in range(B):
        pk = X[b] @ WK  # [T, Hkv*d]
        pv = X[b] @ WV
        for g in range(Hkv):
            KD[b, g, :, slot, :] = pk[:, g * d:(g + 1) * d]
            VD[b, g, :, slot, :] = pv[:, g * d:(g + 1) * d]
    return KD, VD


def sliding_window(kd_hist, vd_hist, window):
    """Bounded slot buffer with a sliding window ("Mixture-of-Depths Attention", closing
    frame: an S << L slot buffer, sliding window variant): of the slots written so far,
    in the order they were written (kd_hist, vd_hist [B,Hkv,T,L,d], slot L-1 the newest),
    a layer reads only the newest `window` ones.  Returns them, oldest first, as float64
    arrays [B,Hkv,T,min(L, window),d]; the joint forward over them is forward(q, k, v,
    *sliding_window(...))."""
    KD, VD = _widen(kd_hist), _widen(vd_hist)
    if KD.ndim != 5 or VD.shape != KD.shape:
        raise ValueError("kd_hist/vd_hist must both be [B,Hkv,T,L,d]")
    if window < 1:
        raise ValueError("window must be >= 1")
    L = KD.shape[3]
    first = max(0, L - window)
    return KD[:, :, :, first:L].copy(), VD[:, :, :, first:L].copy()
