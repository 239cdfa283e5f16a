"""Device-side failure path: a bounded wait that runs out reports MODA_ERR_TIMEOUT
through the status word, the other waits of the CTA leave on its abort flag, and the
CUDA context stays usable (a normal forward afterwards still matches the oracle).
No GPU is hung or faulted: the waits are capped at 20 ms and 2 s."""
import time

import pytest
import torch

from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300.inputs import Shape, make_inputs
from parity_util import TOL_OUT, as_f64, host_view, max_abs

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_reports_timeout():
    binding.load_library()
    t0 = time.perf_counter()
    status = binding.moda_selftest_wait_timeout(20_000_000)
    elapsed = time.perf_counter() - t0
    assert status == 4, binding.STATUS_NAMES.get(status, status)  # MODA_ERR_TIMEOUT
    assert elapsed < 1.5  # the second warp left on the abort flag, not on its 2 s cap
    assert binding.moda_device_status() == 0  # the self-test cleared what it recorded


def test_context_usable_after_timeout(oracle_mod):
    binding.moda_selftest_wait_timeout(5_000_000)
    shape = Shape("after_timeout", 1, 2, 2, 300, 128, 3, torch.bfloat16)
    x = make_inputs(shape, seed=7)
    g = {k: v.cuda() for k, v in x.items()}
    o, lse = binding.moda_fwd(g["q"], g["k"], g["v"], g["kd"], g["vd"])
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    ro, rl = oracle_mod.forward(*(host_view(x[n]) for n in ("q", "k", "v", "kd", "vd")))
    assert max_abs(as_f64(o), ro) < TOL_OUT[torch.bfloat16]
    assert max_abs(as_f64(lse), rl) < TOL_OUT[torch.bfloat16]
