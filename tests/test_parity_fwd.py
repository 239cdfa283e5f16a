"""GPU forward parity: libmoda's moda_fwd (through the C ABI) against the float64 oracle.

Small cases are compared element by element on every output; they span several
128-row tiles with ragged tails, GQA group sizes 1..8, d = 64 and 128, and the
degenerate cases (S = 0, T = 1, T below one tile).  The full-size workloads
are compared on sampled rows the oracle computes one by one.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import WORKLOADS, SEEDS, Shape, make_inputs
from parity_util import TOL_OUT, as_f64, host_view, max_abs, sample_rows

pytestmark = pytest.mark.gpu

f32, bf16 = torch.float32, torch.bfloat16

SMALL = [
    # name, B, H, Hkv, T, d, S, dtype
    ("fp32_small_exact", 1, 2, 2, 256, 64, 4, f32),
    ("fp32_d128_ragged", 1, 4, 2, 200, 128, 5, f32),
    ("bf16_d128_g1_ragged", 1, 2, 2, 300, 128, 8, bf16),
    ("bf16_d128_g4", 2, 8, 2, 260, 128, 24, bf16),
    ("bf16_d64_g4", 1, 8, 2, 384, 64, 32, bf16),
    ("bf16_d64_g2_ragged", 2, 4, 2, 333, 64, 6, bf16),
    ("bf16_no_depth", 1, 4, 4, 257, 128, 0, bf16),
    ("bf16_no_depth_d64", 1, 4, 2, 200, 64, 0, bf16),
    ("bf16_t1", 2, 4, 1, 1, 64, 3, bf16),
    ("bf16_t7", 1, 2, 1, 7, 128, 1, bf16),
    ("bf16_g8", 1, 16, 2, 200, 128, 2, bf16),
    ("bf16_one_slot_long", 1, 4, 1, 1024, 128, 1, bf16),
    ("bf16_g16_d64", 1, 16, 1, 130, 64, 4, bf16),
    # more work units than SMs, so a CTA runs several; the last unit of every (b, kv head)
    # has an empty second query tile (T is not a multiple of the unit's two tiles)
    ("bf16_d64_g1_units_gt_sms", 2, 16, 16, 1100, 64, 4, bf16),
    ("bf16_d64_g4_units_gt_sms", 3, 16, 4, 1100, 64, 8, bf16),
    ("bf16_d128_g1_units_gt_sms", 2, 16, 16, 1100, 128, 4, bf16),
    # more than 128 slots read: the depth keys take two depth steps of one position each
    ("bf16_d64_g4_slots_gt_tile", 1, 8, 2, 200, 64, 160, bf16),
    ("bf16_d128_g2_slots_gt_tile", 1, 4, 2, 150, 128, 130, bf16),
    # G = 1 and 160 slots: 128 one-position chunks per depth step, two depth steps
    ("bf16_d64_g1_slots_gt_tile", 1, 2, 2, 150, 64, 160, bf16),
    # G = 3: 126 of a tile's 128 rows in use, depth chunks of 5 positions (15 rows)
    ("bf16_d64_g3_s24", 1, 6, 2, 300, 64, 24, bf16),
]


def run_fwd(x):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in x.items()}
    o, lse = binding.moda_fwd(g["q"], g["k"], g["v"], g["kd"], g["vd"])
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_forward_small_elementwise(case):
    name, B, H, Hkv, T, d, S, dt = case
    shape = Shape(name, B, H, Hkv, T, d, S, dt)
    x = make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 1)
    o, lse = run_fwd(x)
    ro, rl = oracle.forward(*(host_view(x[n]) for n in ("q", "k", "v", "kd", "vd")))
    tol = TOL_OUT[dt]
    assert np.isfinite(as_f64(o)).all() and np.isfinite(as_f64(lse)).all()
    assert max_abs(as_f64(o), ro) < tol, max_abs(as_f64(o), ro)
    assert max_abs(as_f64(lse), rl) < tol, max_abs(as_f64(lse), rl)


def test_forward_constant_values_give_that_constant():
    """Closed form: with every v and vd equal to c the output is c."""
    shape = Shape("const", 1, 8, 2, 300, 128, 6, bf16)
    x = make_inputs(shape, seed=3)
    c = torch.linspace(-1.5, 2.0, 128).to(bf16)
    x["v"][:] = c
    x["vd"][:] = c
    o, _ = run_fwd(x)
    assert max_abs(as_f64(o), np.broadcast_to(c.float().numpy(), o.shape)) < 1e-2


@pytest.mark.parametrize("name", ["fp32_small", "bf16_mha", "bf16_gqa", "bf16_long", "bf16_train"])
def test_forward_full_size_sampled(name):
    shape = WORKLOADS[name]
    x = make_inputs(shape, seed=SEEDS[name], device="cuda", with_dout=False)
    o, lse = binding.moda_fwd(x["q"], x["k"], x["v"], x["kd"], x["vd"])
    torch.cuda.synchronize()
    rows = sample_rows(shape, 48, seed=SEEDS[name])
    hx = [host_view(x[n]) for n in ("q", "k", "v", "kd", "vd")]
    ro, rl = oracle.forward(*hx, rows=rows)
    go = as_f64(o.reshape(-1, shape.d)[torch.from_numpy(rows).cuda()])
    gl = as_f64(lse.reshape(-1)[torch.from_numpy(rows).cuda()])
    tol = TOL_OUT[shape.dtype]
    assert max_abs(go, ro) < tol, max_abs(go, ro)
    assert max_abs(gl, rl) < tol, max_abs(gl, rl)
    # every output finite, and lse at least the log of the number of visible keys' minimum mass
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_forward_is_deterministic_and_sync_status_clean(monkeypatch):
    shape = Shape("det", 1, 8, 2, 515, 64, 7, bf16)
    x = make_inputs(shape, seed=9)
    o1, l1 = run_fwd(x)
    monkeypatch.setenv("MODA_SYNC", "1")
    o2, l2 = run_fwd(x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert binding.moda_device_status() == 0
