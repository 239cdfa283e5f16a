"""GPU backward parity: libmoda's moda_bwd (through the C ABI) against the float64 oracle.

Small cases: every gradient element compared (relative max error per tensor).
The full-size workloads: sampled positions (dq of the G heads, dkd, dvd)
and sampled sequence keys (dk, dv), which the oracle computes one by one.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import WORKLOADS, SEEDS, Shape, make_inputs
from parity_util import TOL_GRAD_REL, as_f64, host_view, rel_err, sample_keys, sample_positions

pytestmark = pytest.mark.gpu

f32, bf16 = torch.float32, torch.bfloat16
NAMES = ("q", "k", "v", "kd", "vd", "dout")

SMALL = [
    ("fp32_small_exact", 1, 2, 2, 256, 64, 4, f32),
    ("bf16_d64_g4", 1, 4, 1, 300, 64, 5, bf16),
    ("bf16_d128_g1", 1, 2, 2, 260, 128, 3, bf16),
    ("bf16_d64_g4_train_like", 2, 8, 2, 384, 64, 32, bf16),
    ("bf16_d128_g4", 1, 8, 2, 200, 128, 8, bf16),
    ("bf16_no_depth", 1, 4, 2, 257, 64, 0, bf16),
    ("bf16_t1", 1, 4, 2, 1, 64, 2, bf16),
    ("bf16_t9", 1, 2, 1, 9, 128, 1, bf16),
    # d = 64 tensor-core kernels (128-wide tiles): G = 3 leaves 2 padding rows per tile,
    # G = 8, and more CTAs than SMs
    ("bf16_d64_g3_ragged", 1, 6, 2, 300, 64, 5, bf16),
    ("bf16_d64_g8", 1, 16, 2, 260, 64, 3, bf16),
    ("bf16_d64_g1_ctas_gt_sms", 2, 16, 16, 700, 64, 4, bf16),
    # more row blocks than SMs, so the persistent dQ CTAs take several blocks each (blocks of
    # different lengths, the next block's Q/dO staged while one runs): d = 128 with G = 1 and
    # G = 4, and d = 64 with G = 4
    ("bf16_d128_g1_blocks_gt_sms", 2, 16, 16, 700, 128, 4, bf16),
    ("bf16_d128_g4_blocks_gt_sms", 2, 16, 4, 1100, 128, 3, bf16),
    ("bf16_d64_g4_blocks_gt_sms", 2, 16, 4, 1100, 64, 3, bf16),
    # more than 128 slots read (the forward takes two depth key steps)
    ("bf16_d64_g4_slots_gt_tile", 1, 4, 1, 150, 64, 160, bf16),
]


def run(x):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in x.items()}
    o, lse = binding.moda_fwd(g["q"], g["k"], g["v"], g["kd"], g["vd"])
    grads = binding.moda_bwd(g["q"], g["k"], g["v"], g["kd"], g["vd"], o, lse, g["dout"])
    torch.cuda.synchronize()
    return grads


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_backward_small_elementwise(case):
    name, B, H, Hkv, T, d, S, dt = case
    shape = Shape(name, B, H, Hkv, T, d, S, dt, backward=True)
    x = make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 11)
    grads = run(x)
    ref = oracle.backward(*(host_view(x[n]) for n in NAMES))
    for nm, g, r in zip(("dq", "dk", "dv", "dkd", "dvd"), grads, ref):
        if S == 0 and nm in ("dkd", "dvd"):
            continue
        gg = as_f64(g)
        assert np.isfinite(gg).all(), nm
        assert rel_err(gg, r) < TOL_GRAD_REL, (nm, rel_err(gg, r))


@pytest.mark.parametrize("name", ["bf16_train", "bf16_mha", "bf16_gqa"])
def test_backward_full_size_sampled(name):
    # the d = 64 kernels (bf16_train) and the d = 128 ones (bf16_mha: G = 1, bf16_gqa: G = 4)
    shape = WORKLOADS[name]
    x = make_inputs(shape, seed=SEEDS[name], device="cuda", with_dout=True)
    o, lse = binding.moda_fwd(x["q"], x["k"], x["v"], x["kd"], x["vd"])
    dq, dk, dv, dkd, dvd = binding.moda_bwd(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, x["dout"])
    torch.cuda.synchronize()
    hx = [host_view(x[n]) for n in NAMES]
    G, T, d = shape.G, shape.T, shape.d
    pos = sample_positions(shape, 24, seed=5)
    rdq, rdkd, rdvd = oracle.backward_positions(*hx, positions=pos)
    gdq, gdkd, gdvd = [], [], []
    for p in pos:
        t, bg = int(p % T), int(p // T)
        b, g = bg // shape.Hkv, bg % shape.Hkv
        gdq.append(as_f64(dq[b, g * G:(g + 1) * G, t]))
        gdkd.append(as_f64(dkd[b, g, t]))
        gdvd.append(as_f64(dvd[b, g, t]))
    assert rel_err(np.stack(gdq), rdq) < TOL_GRAD_REL
    assert rel_err(np.stack(gdkd), rdkd) < TOL_GRAD_REL
    assert rel_err(np.stack(gdvd), rdvd) < TOL_GRAD_REL
    keys = sample_keys(shape, 6, seed=6)
    rdk, rdv = oracle.backward_keys(*hx, keys=keys)
    idx = torch.from_numpy(keys).cuda()
    assert rel_err(as_f64(dk.reshape(-1, d)[idx]), rdk) < TOL_GRAD_REL
    assert rel_err(as_f64(dv.reshape(-1, d)[idx]), rdv) < TOL_GRAD_REL
    # property that holds at any size: sum_j dk_j + sum_{t,i} dkd_{t,i} = 0 per (b, g)
    tot = dk.double().sum(dim=2) + dkd.double().sum(dim=(2, 3))
    scale_ref = dk.double().abs().sum(dim=2)
    assert float((tot.abs() / scale_ref).max()) < 2e-2


def test_ring_half_full_size_sampled():
    """The training shape while a 32-slot ring is half full (16 slots read of 32 in memory),
    forward and backward at full size on sampled rows, positions and keys; the unread half
    of every position holds NaN, which must not reach any output."""
    shape = WORKLOADS["bf16_train_ring_half"]
    x = make_inputs(shape, seed=SEEDS["bf16_train_ring_half"], device="cuda", with_dout=True)
    S, C = shape.S, shape.S_mem
    x["kd"][:, :, :, S:] = float("nan")
    x["vd"][:, :, :, S:] = float("nan")
    o, lse = binding.moda_fwd(x["q"], x["k"], x["v"], x["kd"], x["vd"], slots=S)
    dq, dk, dv, dkd, dvd = binding.moda_bwd(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, x["dout"], slots=S)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    for t in (o, lse, dq, dk, dv, dkd, dvd):
        assert torch.isfinite(t.float()).all()
    assert bool((dkd[:, :, :, S:] == 0).all()) and bool((dvd[:, :, :, S:] == 0).all())
    read = {n: x[n][:, :, :, :S].contiguous() for n in ("kd", "vd")}
    hx = [host_view(x[n]) if n not in read else host_view(read[n]) for n in NAMES]
    from parity_util import TOL_OUT, max_abs, sample_rows

    rows = sample_rows(shape, 24, seed=7)
    ro, rl = oracle.forward(*hx[:5], rows=rows)
    idx = torch.from_numpy(rows).cuda()
    assert max_abs(as_f64(o.reshape(-1, shape.d)[idx]), ro) < TOL_OUT[shape.dtype]
    assert max_abs(as_f64(lse.reshape(-1)[idx]), rl) < TOL_OUT[shape.dtype]
    G, T = shape.G, shape.T
    pos = sample_positions(shape, 12, seed=8)
    rdq, rdkd, rdvd = oracle.backward_positions(*hx, positions=pos)
    gdq, gdkd, gdvd = [], [], []
    for p in pos:
        t, bg = int(p % T), int(p // T)
        b, g = bg // shape.Hkv, bg % shape.Hkv
        gdq.append(as_f64(dq[b, g * G:(g + 1) * G, t]))
        gdkd.append(as_f64(dkd[b, g, t, :S]))
        gdvd.append(as_f64(dvd[b, g, t, :S]))
    assert rel_err(np.stack(gdq), rdq) < TOL_GRAD_REL
    assert rel_err(np.stack(gdkd), rdkd) < TOL_GRAD_REL
    assert rel_err(np.stack(gdvd), rdvd) < TOL_GRAD_REL
    keys = sample_keys(shape, 3, seed=9)
    rdk, rdv = oracle.backward_keys(*hx, keys=keys)
    kidx = torch.from_numpy(keys).cuda()
    assert rel_err(as_f64(dk.reshape(-1, shape.d)[kidx]), rdk) < TOL_GRAD_REL
    assert rel_err(as_f64(dv.reshape(-1, shape.d)[kidx]), rdv) < TOL_GRAD_REL
