"""GPU parity of the bounded slot buffer (sliding window of depth slots) against the oracle.

A ring of C slots per position is filled on the GPU the way a model would fill it: the
w-th write of the history goes to slot w mod C (moda_depth_store_kv for bf16).  The
forward, backward and decode then read the first S = min(writes, C) ring slots
(slot_capacity = C, S read).  The oracle computes the same step on the sliding window of
the history (its newest C slots, oldest first), so the comparison also checks that the
ring order does not matter.  Slots never written hold large finite junk: were they read,
they would dominate the softmax.  dkd/dvd of those slots must come back exactly zero.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import Shape, make_inputs
from parity_util import TOL_GRAD_REL, TOL_OUT, as_f64, host_view, max_abs, rel_err

pytestmark = pytest.mark.gpu

f32, bf16 = torch.float32, torch.bfloat16

CASES = [
    # name, B, H, Hkv, T, d, C (slots in memory), writes, dtype
    ("bf16_d64_g4_filling", 1, 8, 2, 300, 64, 8, 3, bf16),
    ("bf16_d128_g1_wrapped", 1, 4, 4, 257, 128, 6, 11, bf16),
    ("bf16_d64_g2_just_full", 2, 4, 2, 130, 64, 5, 5, bf16),
    ("bf16_d128_g8_c48_filling", 1, 16, 2, 200, 128, 48, 17, bf16),
    ("bf16_d64_g1_one_of_32", 1, 2, 2, 200, 64, 32, 1, bf16),
    ("bf16_d64_g4_c32_wrapped", 2, 8, 2, 384, 64, 32, 45, bf16),
    ("fp32_d64_g2_filling", 1, 4, 2, 100, 64, 6, 4, f32),
]


def ring_slot_of_window(n_writes, C):
    """Ring slot holding each window entry (window entry i is write n - S + i)."""
    S = min(n_writes, C)
    return [(n_writes - S + i) % C for i in range(S)]


def build_ring(hist_k, hist_v, C, junk=8.0):
    """Fills a [B,Hkv,T,C,d] ring on the GPU with the history's writes in order."""
    B, Hkv, T, n, d = hist_k.shape
    ring_k = torch.full((B, Hkv, T, C, d), junk, dtype=hist_k.dtype, device="cuda")
    ring_v = torch.full((B, Hkv, T, C, d), -junk, dtype=hist_k.dtype, device="cuda")
    for w in range(n):
        hk = hist_k[:, :, :, w].contiguous().cuda()
        hv = hist_v[:, :, :, w].contiguous().cuda()
        if hist_k.dtype == bf16:
            binding.moda_depth_store_kv(hk, hv, ring_k, ring_v, w % C)
        else:
            ring_k[:, :, :, w % C] = hk
            ring_v[:, :, :, w % C] = hv
    return ring_k, ring_v


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ring_forward_backward(case):
    name, B, H, Hkv, T, d, C, n, dt = case
    shape = Shape(name, B, H, Hkv, T, d, n, dt, backward=True)
    x = make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 51)  # kd/vd = the write history
    S = min(n, C)
    ring_k, ring_v = build_ring(x["kd"], x["vd"], C)
    g = {nm: x[nm].cuda() for nm in ("q", "k", "v", "dout")}
    o, lse = binding.moda_fwd(g["q"], g["k"], g["v"], ring_k, ring_v, slots=S)
    dq, dk, dv, dkd, dvd = binding.moda_bwd(g["q"], g["k"], g["v"], ring_k, ring_v, o, lse, g["dout"], slots=S)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0

    wk, wv = oracle.sliding_window(host_view(x["kd"]), host_view(x["vd"]), C)
    hq, hk, hv, hd = (as_f64(x[nm]) for nm in ("q", "k", "v", "dout"))  # exact widening, like the window
    ro, rl = oracle.forward(hq, hk, hv, wk, wv)
    assert max_abs(as_f64(o), ro) < TOL_OUT[dt], max_abs(as_f64(o), ro)
    assert max_abs(as_f64(lse), rl) < TOL_OUT[dt], max_abs(as_f64(lse), rl)

    rdq, rdk, rdv, rdkd, rdvd = oracle.backward(hq, hk, hv, wk, wv, hd)
    for nm, got, ref in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
        assert rel_err(as_f64(got), ref) < TOL_GRAD_REL, (nm, rel_err(as_f64(got), ref))
    slots = ring_slot_of_window(n, C)
    for nm, got, ref in (("dkd", dkd, rdkd), ("dvd", dvd, rdvd)):
        gg = as_f64(got)
        assert rel_err(gg[:, :, :, slots], ref) < TOL_GRAD_REL, (nm, rel_err(gg[:, :, :, slots], ref))
        unread = [s for s in range(C) if s not in slots]
        if unread:
            assert np.all(gg[:, :, :, unread] == 0.0), nm


NAN_CASES = [
    # name, B, H, Hkv, T, d, C (slots in memory), S read, dtype
    ("bf16_d64_g4_half", 1, 8, 2, 300, 64, 32, 16, bf16),
    ("bf16_d128_g1_third", 1, 4, 4, 257, 128, 24, 8, bf16),
    ("bf16_d128_g4_one", 2, 8, 2, 200, 128, 8, 1, bf16),
    ("fp32_d64_g2_half", 1, 4, 2, 100, 64, 6, 3, f32),
]


@pytest.mark.parametrize("case", NAN_CASES, ids=[c[0] for c in NAN_CASES])
def test_unread_slots_holding_nan_and_inf_change_nothing(case):
    """Slots S .. C-1 of a bounded slot buffer are outside the layer's depth memory: the
    forward and the backward must not read them.  They are filled with NaN (keys) and
    +/-Inf (values), which would poison any sum they entered, even with zero weight."""
    name, B, H, Hkv, T, d, C, S, dt = case
    shape = Shape(name, B, H, Hkv, T, d, S, dt, backward=True)
    x = make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 71)
    ring_k = torch.full((B, Hkv, T, C, d), float("nan"), dtype=dt)
    ring_v = torch.full((B, Hkv, T, C, d), float("inf"), dtype=dt)
    ring_v[..., ::2] = float("-inf")
    ring_k[:, :, :, :S] = x["kd"]
    ring_v[:, :, :, :S] = x["vd"]
    g = {nm: x[nm].cuda() for nm in ("q", "k", "v", "dout")}
    rk, rv = ring_k.cuda(), ring_v.cuda()
    o, lse = binding.moda_fwd(g["q"], g["k"], g["v"], rk, rv, slots=S)
    dq, dk, dv, dkd, dvd = binding.moda_bwd(g["q"], g["k"], g["v"], rk, rv, o, lse, g["dout"], slots=S)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    hx = [host_view(x[nm]) for nm in ("q", "k", "v", "kd", "vd", "dout")]
    ro, rl = oracle.forward(*hx[:5])
    assert np.isfinite(as_f64(o)).all() and np.isfinite(as_f64(lse)).all()
    assert max_abs(as_f64(o), ro) < TOL_OUT[dt], max_abs(as_f64(o), ro)
    assert max_abs(as_f64(lse), rl) < TOL_OUT[dt], max_abs(as_f64(lse), rl)
    ref = oracle.backward(*hx)
    for nm, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref[:3]):
        assert rel_err(as_f64(got), r) < TOL_GRAD_REL, (nm, rel_err(as_f64(got), r))
    for nm, got, r in (("dkd", dkd, ref[3]), ("dvd", dvd, ref[4])):
        gg = as_f64(got)
        assert rel_err(gg[:, :, :, :S], r) < TOL_GRAD_REL, (nm, rel_err(gg[:, :, :, :S], r))
        assert np.all(gg[:, :, :, S:] == 0.0), nm


@pytest.mark.parametrize("case", [c for c in CASES if c[-1] == bf16], ids=[c[0] for c in CASES if c[-1] == bf16])
def test_ring_decode(case):
    """The decode step of the newest position reads the same ring (its slots [B,Hkv,C,d])."""
    name, B, H, Hkv, T, d, C, n, dt = case
    shape = Shape(name, B, H, Hkv, T, d, n, dt)
    x = make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 61)
    S = min(n, C)
    ring_k, ring_v = build_ring(x["kd"], x["vd"], C)
    q_new = x["q"][:, :, T - 1].contiguous()
    o, lse = binding.moda_decode(q_new.cuda(), x["k"].cuda(), x["v"].cuda(), ring_k[:, :, T - 1].contiguous(),
                                 ring_v[:, :, T - 1].contiguous(), slots=S)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    wk, wv = oracle.sliding_window(host_view(x["kd"]), host_view(x["vd"]), C)
    ro, rl = oracle.decode(as_f64(q_new), as_f64(x["k"]), as_f64(x["v"]), wk[:, :, T - 1], wv[:, :, T - 1])
    assert max_abs(as_f64(o), ro) < TOL_OUT[bf16], max_abs(as_f64(o), ro)
    assert max_abs(as_f64(lse), rl) < TOL_OUT[bf16], max_abs(as_f64(lse), rl)


@pytest.mark.parametrize("case", [c for c in NAN_CASES if c[-1] == bf16], ids=[c[0] for c in NAN_CASES if c[-1] == bf16])
def test_decode_unread_slots_holding_nan_and_inf_change_nothing(case):
    """The decode step reads only slots 0 .. S-1 of the newest position's ring; the others,
    NaN (keys) and +/-Inf (values), enter no product (0 * NaN would poison one)."""
    name, B, H, Hkv, T, d, C, S, dt = case
    shape = Shape(name, B, H, Hkv, T, d, S, dt)
    x = make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 81)
    ring_k = torch.full((B, Hkv, C, d), float("nan"), dtype=dt)
    ring_v = torch.full((B, Hkv, C, d), float("inf"), dtype=dt)
    ring_v[..., ::2] = float("-inf")
    ring_k[:, :, :S] = x["kd"][:, :, T - 1]
    ring_v[:, :, :S] = x["vd"][:, :, T - 1]
    q_new = x["q"][:, :, T - 1].contiguous()
    o, lse = binding.moda_decode(q_new.cuda(), x["k"].cuda(), x["v"].cuda(), ring_k.cuda(), ring_v.cuda(), slots=S)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    ro, rl = oracle.decode(as_f64(q_new), as_f64(x["k"]), as_f64(x["v"]), as_f64(x["kd"][:, :, T - 1]),
                           as_f64(x["vd"][:, :, T - 1]))
    assert np.isfinite(as_f64(o)).all() and np.isfinite(as_f64(lse)).all()
    assert max_abs(as_f64(o), ro) < TOL_OUT[dt], max_abs(as_f64(o), ro)
    assert max_abs(as_f64(lse), rl) < TOL_OUT[dt], max_abs(as_f64(lse), rl)


def test_ring_rejects_capacity_below_slots():
    """slot_capacity below S is an argument error (nothing launched)."""
    q = torch.zeros(1, 2, 8, 64, dtype=bf16, device="cuda")
    k = torch.zeros(1, 2, 8, 64, dtype=bf16, device="cuda")
    kd = torch.zeros(1, 2, 8, 4, 64, dtype=bf16, device="cuda")
    with pytest.raises(binding.MODAError):
        binding.moda_fwd(q, k, k, kd, kd, slots=5)
