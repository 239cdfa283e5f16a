"""GPU decode parity: libmoda's moda_decode (through the C ABI) against the float64 oracle.

Small cases are compared element by element: T = 1, S = 0, ragged key counts around the
128-key sub-tile, GQA groups 1..8, d = 64 and 128, many key splits, and a cache whose
capacity exceeds T with NaN in the unused positions (they must not leak into the step).
The full-size decode workloads are compared on sampled (batch, kv head) groups, and the
step is checked against row T-1 of moda_fwd on the same inputs.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import DECODE_SEEDS, DECODE_WORKLOADS, Shape, make_decode_inputs
from parity_util import TOL_OUT, as_f64, host_view, max_abs

pytestmark = pytest.mark.gpu

bf16 = torch.bfloat16

SMALL = [
    # name, B, H, Hkv, T, d, S, capacity
    ("t1_no_depth", 1, 2, 2, 1, 64, 0, 1),
    ("t1_depth", 2, 4, 1, 1, 128, 3, 1),
    ("d128_g4", 2, 8, 2, 300, 128, 5, 300),
    ("d64_g1_ragged", 1, 4, 4, 129, 64, 3, 129),
    ("d128_g8_long_depth", 2, 16, 2, 1000, 128, 48, 1000),
    ("d64_g3_no_depth", 1, 6, 2, 257, 64, 0, 257),
    ("d64_g2_capacity_nan_tail", 2, 4, 2, 777, 64, 7, 1024),
    ("d128_g4_many_splits", 1, 8, 2, 9000, 128, 2, 9000),
    ("d64_g5_depth_over_128", 1, 5, 1, 200, 64, 200, 200),
]


def run_decode(x, T, S):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in x.items()}
    o, lse = binding.moda_decode(g["q"], g["k"], g["v"], g["kd"] if S else None, g["vd"] if S else None, T=T)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    return o, lse


def oracle_decode(x, T):
    return oracle.decode(host_view(x["q"]), host_view(x["k"][:, :, :T]), host_view(x["v"][:, :, :T]),
                         host_view(x["kd"]), host_view(x["vd"]))


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_decode_small_elementwise(case):
    name, B, H, Hkv, T, d, S, cap = case
    shape = Shape(name, B, H, Hkv, T, d, S, bf16)
    x = make_decode_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 21, capacity=cap)
    if cap > T:
        x["k"][:, :, T:] = float("nan")
        x["v"][:, :, T:] = float("nan")
    o, lse = run_decode(x, T, S)
    ro, rl = oracle_decode(x, T)
    assert np.isfinite(as_f64(o)).all() and np.isfinite(as_f64(lse)).all()
    assert max_abs(as_f64(o), ro) < TOL_OUT[bf16], max_abs(as_f64(o), ro)
    assert max_abs(as_f64(lse), rl) < TOL_OUT[bf16], max_abs(as_f64(lse), rl)


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_full_size_sampled(name):
    """The whole step on the GPU; the oracle recomputes a few (batch, kv head) groups."""
    shape = DECODE_WORKLOADS[name]
    x = make_decode_inputs(shape, seed=DECODE_SEEDS[name], device="cuda")
    o, lse = binding.moda_decode(x["q"], x["k"], x["v"], x["kd"], x["vd"])
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    rng = np.random.default_rng(9)
    G = shape.G
    for _ in range(3):
        b, g = int(rng.integers(shape.B)), int(rng.integers(shape.Hkv))
        sub = {"q": x["q"][b:b + 1, g * G:(g + 1) * G], "k": x["k"][b:b + 1, g:g + 1], "v": x["v"][b:b + 1, g:g + 1],
               "kd": x["kd"][b:b + 1, g:g + 1], "vd": x["vd"][b:b + 1, g:g + 1]}
        ro, rl = oracle_decode({k: v.cpu() for k, v in sub.items()}, shape.T)
        go = as_f64(o[b:b + 1, g * G:(g + 1) * G])
        gl = as_f64(lse[b:b + 1, g * G:(g + 1) * G])
        assert max_abs(go, ro) < TOL_OUT[bf16], (name, b, g, max_abs(go, ro))
        assert max_abs(gl, rl) < TOL_OUT[bf16], (name, b, g, max_abs(gl, rl))


def test_decode_is_forward_last_row():
    """moda_decode equals row T-1 of moda_fwd when the forward's depth slab at T-1 holds the
    decode step's slots (both through the C ABI, within bf16 rounding of either)."""
    B, H, Hkv, T, d, S = 2, 8, 2, 333, 64, 6
    gen = torch.Generator(device="cpu").manual_seed(5)
    q = torch.randn(B, H, T, d, generator=gen).to(bf16).cuda()
    k = torch.randn(B, Hkv, T, d, generator=gen).to(bf16).cuda()
    v = torch.randn(B, Hkv, T, d, generator=gen).to(bf16).cuda()
    kd = torch.randn(B, Hkv, T, S, d, generator=gen).to(bf16).cuda()
    vd = torch.randn(B, Hkv, T, S, d, generator=gen).to(bf16).cuda()
    of, lf = binding.moda_fwd(q, k, v, kd, vd)
    od, ld = binding.moda_decode(q[:, :, T - 1].contiguous(), k, v, kd[:, :, T - 1].contiguous(),
                                 vd[:, :, T - 1].contiguous())
    torch.cuda.synchronize()
    assert max_abs(as_f64(od), as_f64(of[:, :, T - 1])) < 2 * TOL_OUT[bf16]
    assert max_abs(as_f64(ld), as_f64(lf[:, :, T - 1])) < 1e-3


def test_decode_rejects_bad_arguments():
    """Synchronous argument checks: fp32, a capacity below T, a short workspace."""
    q = torch.zeros(1, 2, 64, dtype=torch.float32, device="cuda")
    kc = torch.zeros(1, 2, 8, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.MODAError):
        binding.moda_decode(q, kc, kc, None, None)
    qb, kb = q.to(bf16), kc.to(bf16)
    with pytest.raises(binding.MODAError):
        binding.moda_decode(qb, kb, kb, None, None, T=9)
    with pytest.raises(binding.MODAError):
        binding.moda_decode(qb, kb, kb, None, None, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
