"""GPU parity of the depth-KV write path (moda_depth_store_kv, moda_depth_project_kv through
the C ABI) against the float64 oracle.

The store is a copy, so it must be bit-exact.  The projection sums bf16 products in
float32 and rounds once to bf16, so each element may differ from the float64 value y by
half a bf16 ulp of y plus the float32 summation error; the bound used is
    |gpu - y| <= 2^-8 |y| + Dm * 2^-23 * sum_m |x_m w_m| + 1e-6.
Both operations must leave every slot but the written one, bit for bit, as it was.
Small cases are compared whole (ragged T around the 128-position tile, Hkv*d not a
multiple of the 128-column tile, d_model not a multiple of the 64-wide reduction step,
T = 1, a single slot); the full-size write workloads are compared on sampled
positions, with the untouched-slot check over the whole cache.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import WRITE_SEEDS, WRITE_WORKLOADS, Shape, make_write_inputs
from parity_util import as_f64, host_view

pytestmark = pytest.mark.gpu

bf16 = torch.bfloat16


def _shape(name, B, Hkv, T, S, d):
    return Shape(name, B, Hkv, Hkv, T, d, S, bf16)


def _proj_bound(x, w, ref):
    """Elementwise bound for one float32-accumulated, bf16-rounded product x @ w (x [T, Dm],
    w [Dm, N] as float64 arrays of the bf16 inputs) around its float64 value ref."""
    Dm = x.shape[1]
    return 2.0 ** -8 * np.abs(ref) + Dm * 2.0 ** -23 * (np.abs(x) @ np.abs(w)) + 1e-6


def _check_slot_untouched(before, after, slot):
    S = before.shape[3]
    others = [s for s in range(S) if s != slot]
    if others:
        assert torch.equal(before[:, :, :, others], after[:, :, :, others])


STORE_CASES = [
    # name, B, Hkv, T, S, d, slot
    ("t1_one_slot_d64", 1, 1, 1, 1, 64, 0),
    ("d128_ragged_last_slot", 2, 3, 129, 4, 128, 3),
    ("d64_mid_slot", 1, 2, 300, 7, 64, 2),
    ("d64_s32_last", 2, 4, 1000, 32, 64, 31),
]


@pytest.mark.parametrize("case", STORE_CASES, ids=[c[0] for c in STORE_CASES])
def test_store_small_exact(case):
    name, B, Hkv, T, S, d, slot = case
    x = make_write_inputs(_shape(name, B, Hkv, T, S, d), seed=zlib.crc32(name.encode()) % 1000 + 31, Dm=64)
    g = {k: v.cuda() for k, v in x.items()}
    kd0, vd0 = g["kd"].clone(), g["vd"].clone()
    binding.moda_depth_store_kv(g["k"], g["v"], g["kd"], g["vd"], slot)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    rk, rv = oracle.depth_store(host_view(x["k"]), host_view(x["v"]), host_view(x["kd"]), host_view(x["vd"]), slot)
    assert np.array_equal(as_f64(g["kd"]), rk)
    assert np.array_equal(as_f64(g["vd"]), rv)
    _check_slot_untouched(kd0, g["kd"], slot)
    _check_slot_untouched(vd0, g["vd"], slot)


PROJECT_CASES = [
    # name, B, Hkv, T, S, d, Dm, slot
    ("t1_d64_dm64", 1, 1, 1, 1, 64, 64, 0),
    ("d128_ragged_t", 2, 2, 300, 4, 128, 512, 1),
    ("d64_n192_dm200", 1, 3, 129, 2, 64, 200, 0),
    ("d128_n1024", 2, 8, 260, 5, 128, 1024, 4),
    ("d64_dm8", 1, 1, 128, 3, 64, 8, 2),
    ("d64_n64_long_dm", 1, 1, 333, 2, 64, 2056, 1),
]


def _oracle_project_check(x, g, slot):
    """Compares slot `slot` of the GPU's kd/vd with the oracle's projection, element by element."""
    hx = {k: host_view(v) for k, v in x.items()}
    rk, rv = oracle.depth_project(hx["x"], hx["wk"], hx["wv"], hx["kd"], hx["vd"], slot)
    X, WK, WV = as_f64(x["x"]), as_f64(x["wk"]), as_f64(x["wv"])
    B, Hkv, T, S, d = rk.shape
    for name, ref, w in (("kd", rk, WK), ("vd", rv, WV)):
        got = as_f64(g[name])
        others = [s for s in range(S) if s != slot]
        assert np.array_equal(got[:, :, :, others], ref[:, :, :, others])
        for b in range(B):
            bound = _proj_bound(X[b], w, X[b] @ w)  # [T, Hkv*d]
            for gh in range(Hkv):
                err = np.abs(got[b, gh, :, slot] - ref[b, gh, :, slot])
                lim = bound[:, gh * d:(gh + 1) * d]
                assert (err <= lim).all(), (name, b, gh, float(np.max(err - lim)))


@pytest.mark.parametrize("case", PROJECT_CASES, ids=[c[0] for c in PROJECT_CASES])
def test_project_small_elementwise(case):
    name, B, Hkv, T, S, d, Dm, slot = case
    x = make_write_inputs(_shape(name, B, Hkv, T, S, d), seed=zlib.crc32(name.encode()) % 1000 + 41, Dm=Dm)
    g = {k: v.cuda() for k, v in x.items()}
    binding.moda_depth_project_kv(g["x"], g["wk"], g["wv"], g["kd"], g["vd"], slot)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    _oracle_project_check(x, g, slot)


def test_project_then_forward():
    """A slot written by the projection is read by moda_fwd like any other slot: GPU
    projection + GPU forward against oracle projection + oracle forward."""
    B, H, Hkv, T, S, d, Dm, slot = 1, 8, 2, 200, 3, 64, 256, 1
    shape = Shape("feed", B, H, Hkv, T, d, S, bf16)
    x = make_write_inputs(shape, seed=77, Dm=Dm)
    gen = torch.Generator().manual_seed(78)
    q = torch.randn(B, H, T, d, generator=gen).to(bf16)
    g = {k: v.cuda() for k, v in x.items()}
    binding.moda_depth_project_kv(g["x"], g["wk"], g["wv"], g["kd"], g["vd"], slot)
    o, lse = binding.moda_fwd(q.cuda(), g["k"], g["v"], g["kd"], g["vd"])
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    # the oracle reads the GPU's projected slot only through its own projection
    hx = {k: host_view(v) for k, v in x.items()}
    rkd, rvd = oracle.depth_project(hx["x"], hx["wk"], hx["wv"], hx["kd"], hx["vd"], slot)
    # round the oracle's slot to bf16 as the cache stores it, then run the oracle forward
    rkd = torch.from_numpy(rkd).to(bf16)
    rvd = torch.from_numpy(rvd).to(bf16)
    ro, rl = oracle.forward(host_view(q), hx["k"], hx["v"], host_view(rkd), host_view(rvd))
    assert float(np.max(np.abs(as_f64(o) - ro))) < 2e-2
    assert float(np.max(np.abs(as_f64(lse) - rl))) < 2e-2


@pytest.mark.parametrize("name", list(WRITE_WORKLOADS))
def test_write_full_size_sampled(name):
    """Both writes at full size: sampled positions against the oracle, the other slots
    untouched over the whole cache."""
    shape = WRITE_WORKLOADS[name]
    x = make_write_inputs(shape, seed=WRITE_SEEDS[name], device="cuda")
    B, Hkv, T, S, d = shape.B, shape.Hkv, shape.T, shape.S, shape.d
    slot_store, slot_proj = S - 1, S // 2
    kd0, vd0 = x["kd"].clone(), x["vd"].clone()
    binding.moda_depth_store_kv(x["k"], x["v"], x["kd"], x["vd"], slot_store)
    binding.moda_depth_project_kv(x["x"], x["wk"], x["wv"], x["kd"], x["vd"], slot_proj)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    others = [s for s in range(S) if s not in (slot_store, slot_proj)]
    assert torch.equal(kd0[:, :, :, others], x["kd"][:, :, :, others])
    assert torch.equal(vd0[:, :, :, others], x["vd"][:, :, :, others])
    del kd0, vd0
    rng = np.random.default_rng(3)
    ts = np.unique(np.concatenate([[0, 127, 128, T - 1], rng.integers(0, T, 12)]))
    for _ in range(3):
        b, gh = int(rng.integers(B)), int(rng.integers(Hkv))
        sub_k = x["k"][b:b + 1, gh:gh + 1, ts].cpu()
        sub_v = x["v"][b:b + 1, gh:gh + 1, ts].cpu()
        sub_kd = x["kd"][b:b + 1, gh:gh + 1, ts].cpu()
        sub_vd = x["vd"][b:b + 1, gh:gh + 1, ts].cpu()
        rk, rv = oracle.depth_store(host_view(sub_k), host_view(sub_v), host_view(sub_kd), host_view(sub_vd),
                                    slot_store)
        assert np.array_equal(as_f64(sub_kd)[..., slot_store, :], rk[..., slot_store, :])
        assert np.array_equal(as_f64(sub_vd)[..., slot_store, :], rv[..., slot_store, :])
        sx = x["x"][b:b + 1, ts].cpu()
        cols = slice(gh * d, (gh + 1) * d)
        swk, swv = x["wk"][:, cols].cpu(), x["wv"][:, cols].cpu()
        rk, rv = oracle.depth_project(host_view(sx), host_view(swk), host_view(swv), host_view(sub_kd),
                                      host_view(sub_vd), slot_proj)
        X = as_f64(sx)[0]
        for got, ref, w in ((sub_kd, rk, swk), (sub_vd, rv, swv)):
            W = as_f64(w)
            err = np.abs(as_f64(got)[0, 0, :, slot_proj] - ref[0, 0, :, slot_proj])
            assert (err <= _proj_bound(X, W, X @ W)).all(), (name, b, gh)


def test_write_rejects_bad_arguments():
    """Synchronous argument checks: slot out of range, fp32, d_model not a multiple of 8."""
    kd = torch.zeros(1, 1, 4, 2, 64, dtype=bf16, device="cuda")
    k = torch.zeros(1, 1, 4, 64, dtype=bf16, device="cuda")
    with pytest.raises(binding.MODAError):
        binding.moda_depth_store_kv(k, k, kd, kd.clone(), 2)
    with pytest.raises(binding.MODAError):
        binding.moda_depth_store_kv(k.float(), k.float(), kd.float(), kd.float(), 0)
    x = torch.zeros(1, 4, 12, dtype=bf16, device="cuda")
    w = torch.zeros(12, 64, dtype=bf16, device="cuda")
    with pytest.raises(binding.MODAError):
        binding.moda_depth_project_kv(x, w, w, kd, kd.clone(), 0)
