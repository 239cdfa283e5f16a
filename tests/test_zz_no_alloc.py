"""The allocation-free backward entry point (moda_bwd_noalloc).

Some callers cannot allocate device memory at call time (allocator hooks, runtimes
whose device-memory budget is fixed at start-up, plain-C callers with no allocator),
so the library offers moda_bwd without a workspace argument: its scratch is a fixed
array inside the library.  These tests call it through the C ABI twice in a row and
compare each result with moda_bwd given a normal workspace.  The file sorts last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import Shape, make_inputs
from parity_util import TOL_GRAD_REL, as_f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [("bf16_d64_g4", 1, 8, 2, 300, 64, 5, torch.bfloat16),
                                  ("bf16_d128_g1", 2, 2, 2, 200, 128, 3, torch.bfloat16),
                                  ("fp32_d64", 1, 2, 1, 150, 64, 4, torch.float32)],
                         ids=lambda c: c[0])
def test_noalloc_matches_workspace_backward_twice(case):
    name, B, H, Hkv, T, d, S, dt = case
    shape = Shape(name, B, H, Hkv, T, d, S, dt, backward=True)
    x = {k: v.cuda() for k, v in make_inputs(shape, seed=77).items()}
    o, lse = binding.moda_fwd(x["q"], x["k"], x["v"], x["kd"], x["vd"])
    ref = binding.moda_bwd(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, x["dout"])
    torch.cuda.synchronize()
    for _ in range(2):
        grads = tuple(torch.full_like(t, float("nan")) for t in ref)
        binding.moda_bwd_noalloc(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, x["dout"], grads)
        torch.cuda.synchronize()
        for nm, g, r in zip(("dq", "dk", "dv", "dkd", "dvd"), grads, ref):
            ga, ra = as_f64(g), as_f64(r)
            assert np.isfinite(ga).all(), nm
            assert rel_err(ga, ra) < TOL_GRAD_REL, (nm, rel_err(ga, ra))
    assert binding.moda_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_array():
    lib = binding.load_library()
    cap = binding.moda_bwd_noalloc_max_workspace_bytes()
    assert cap == 32 << 20
    big = binding.make_desc(4, 32, 8, 8192, 4, 128, torch.bfloat16)
    assert binding.moda_bwd_workspace_bytes(big) > cap
    fake = [ctypes.c_void_p(1 << 20)] * 13
    assert lib.moda_bwd_noalloc(ctypes.byref(big), *fake, None) == 5  # MODA_ERR_WORKSPACE, nothing launched


def _rows_at_cap(d):
    """B*H*T rows whose workspace (row statistics, then the float32 dq share, each rounded
    up to 256 bytes) is the largest that fits the array."""
    cap = binding.moda_bwd_noalloc_max_workspace_bytes()
    align = lambda n: (n + 255) // 256 * 256  # noqa: E731
    rows = cap // (8 + 4 * d)
    while align(rows * 8) + align(rows * 4 * d) > cap:
        rows -= 1
    return rows


def test_noalloc_at_its_capacity_and_one_row_over():
    """A problem whose workspace fills the array to its last bytes (so an offset or rounding
    error in the workspace layout would touch memory past it) matches moda_bwd with a normal
    workspace on two calls in a row; one more row is refused before anything launches."""
    d, H, Hkv, S = 64, 4, 1, 2
    rows = _rows_at_cap(d)
    assert rows % H == 0
    T = rows // H
    shape = Shape("at_cap", 1, H, Hkv, T, d, S, torch.bfloat16, backward=True)
    desc = binding.make_desc(1, H, Hkv, T, S, d, torch.bfloat16)
    cap = binding.moda_bwd_noalloc_max_workspace_bytes()
    assert cap - 512 < binding.moda_bwd_workspace_bytes(desc) <= cap
    x = make_inputs(shape, seed=78, device="cuda")
    o, lse = binding.moda_fwd(x["q"], x["k"], x["v"], x["kd"], x["vd"])
    ref = binding.moda_bwd(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, x["dout"])
    torch.cuda.synchronize()
    for _ in range(2):
        grads = tuple(torch.full_like(t, float("nan")) for t in ref)
        binding.moda_bwd_noalloc(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, x["dout"], grads)
        torch.cuda.synchronize()
        for nm, g, r in zip(("dq", "dk", "dv", "dkd", "dvd"), grads, ref):
            ga, ra = as_f64(g), as_f64(r)
            assert np.isfinite(ga).all(), nm
            assert rel_err(ga, ra) < TOL_GRAD_REL, (nm, rel_err(ga, ra))
    assert binding.moda_device_status() == 0
    over = binding.make_desc(1, H, Hkv, T + 1, S, d, torch.bfloat16)
    assert binding.moda_bwd_workspace_bytes(over) > cap
    lib = binding.load_library()
    fake = [ctypes.c_void_p(1 << 20)] * 13
    assert lib.moda_bwd_noalloc(ctypes.byref(over), *fake, None) == 5  # MODA_ERR_WORKSPACE, nothing launched
