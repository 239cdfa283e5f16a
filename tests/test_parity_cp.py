"""GPU parity of the context-parallel pieces (moda_fwd_partial, moda_merge_partial,
moda_bwd_partial, moda_convert_f32) against the unchunked float64 oracle.

A problem is cut into chunks on one GPU; every rank of the ring schedule runs in turn
in this process (no kernel waits on another), each pair goes through the library, and
the assembled outputs and gradients are compared element by element with the oracle's
unchunked forward and backward.  A second family cuts the key range of each query chunk
at random places, so the pairs have partly visible key tiles, key ranges that are not
multiples of a tile and offsets that are not chunk-aligned.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from joint_sequence_depth_gb300 import binding
from joint_sequence_depth_gb300 import context_parallel as cp
from joint_sequence_depth_gb300.inputs import Shape, make_inputs
from parity_util import TOL_GRAD_REL, TOL_OUT, as_f64, host_view, max_abs, rel_err

pytestmark = pytest.mark.gpu

bf16, f32 = torch.bfloat16, torch.float32
NAMES = ("q", "k", "v", "kd", "vd", "dout")

RING = [
    # name, B, H, Hkv, T, d, S, dtype, world, layout
    ("d128_g4_w2", 1, 8, 2, 600, 128, 6, bf16, 2, "contiguous"),
    ("d64_g1_w3_ragged", 2, 4, 4, 517, 64, 4, bf16, 3, "contiguous"),
    ("d64_g4_w4_zigzag", 1, 8, 2, 1000, 64, 8, bf16, 4, "zigzag"),
    ("d128_g8_w2_zigzag", 1, 16, 2, 390, 128, 2, bf16, 2, "zigzag"),
    ("d64_g2_no_depth_w3", 1, 4, 2, 700, 64, 0, bf16, 3, "contiguous"),
    ("fp32_d64_w2", 1, 4, 2, 300, 64, 3, f32, 2, "zigzag"),
    # G = 16: the bf16 backward of every pair runs on the CUDA cores (float32 accumulators)
    ("d64_g16_w2_cuda_core_bwd", 1, 16, 1, 300, 64, 2, bf16, 2, "contiguous"),
]


def _split(t, chunks):
    return [t.narrow(2, c.start, c.length).contiguous() for c in chunks]


def _assemble(parts, chunks, T):
    shape = list(parts[0].shape)
    shape[2] = T
    out = torch.empty(shape, dtype=parts[0].dtype, device=parts[0].device)
    for p, c in zip(parts, chunks):
        out.narrow(2, c.start, c.length).copy_(p)
    return out


def _inputs(name, B, H, Hkv, T, d, S, dt):
    shape = Shape(name, B, H, Hkv, T, d, S, dt, backward=True)
    return make_inputs(shape, seed=zlib.crc32(name.encode()) % 1000 + 21)


@pytest.mark.parametrize("case", RING, ids=[c[0] for c in RING])
def test_ring_schedule_on_one_gpu_matches_the_unchunked_oracle(case):
    name, B, H, Hkv, T, d, S, dt, world, layout = case
    x = _inputs(name, B, H, Hkv, T, d, S, dt)
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in NAMES}
    owned = cp.chunks_of(T, world, layout)
    depth = S > 0
    loc = {n: [(_split(g[n], owned[r]) if (depth or n not in ("kd", "vd")) else [None] * len(owned[r]))
               for r in range(world)] for n in NAMES}
    o, lse = cp.simulate_ring_forward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], T, world, layout)
    grads = cp.simulate_ring_backward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], o, lse, loc["dout"], T,
                                      world, layout)
    torch.cuda.synchronize()
    assert binding.moda_device_status() == 0
    chunks = [c for cs in owned for c in cs]
    flat = lambda per_rank: [p for r in range(world) for p in per_rank[r]]  # noqa: E731
    go, gl = _assemble(flat(o), chunks, T), _assemble(flat(lse), chunks, T)
    hx = [host_view(x[n]) for n in NAMES]
    ro, rl = oracle.forward(*hx[:5])
    tol = TOL_OUT[dt]
    assert max_abs(as_f64(go), ro) < tol, max_abs(as_f64(go), ro)
    assert max_abs(as_f64(gl), rl) < tol, max_abs(as_f64(gl), rl)
    ref = oracle.backward(*hx)
    for i, nm in enumerate(("dq", "dk", "dv", "dkd", "dvd")):
        if not depth and nm in ("dkd", "dvd"):
            continue
        got = as_f64(_assemble(flat(grads[i]), chunks, T))
        assert np.isfinite(got).all(), nm
        assert rel_err(got, ref[i]) < TOL_GRAD_REL, (nm, rel_err(got, ref[i]))


SPLITS = [
    # name, B, H, Hkv, T, d, S, dtype: query chunks and key pieces cut at random places
    ("split_d128_g2", 1, 4, 2, 700, 128, 5, bf16),
    ("split_d64_g4", 2, 8, 2, 650, 64, 3, bf16),
    ("split_d64_g1_no_depth", 1, 2, 2, 900, 64, 0, bf16),
    ("split_d128_g8", 1, 16, 2, 450, 128, 8, bf16),
    ("split_fp32_d128", 1, 4, 4, 300, 128, 2, f32),
]


def _random_tiling(T, seed):
    """Query chunks [q0, q1) at random cuts; for each, key pieces that partition [0, q1),
    every piece starting at or before q0 (the geometry moda_fwd_partial accepts)."""
    rng = np.random.default_rng(seed)
    cuts = sorted(set(rng.integers(1, T, size=3).tolist()))
    bounds = [0] + cuts + [T]
    tiles = []
    for q0, q1 in zip(bounds[:-1], bounds[1:]):
        kc = sorted(set(rng.integers(1, q0 + 1, size=3).tolist())) if q0 > 0 else []
        kb = [0] + kc + [q1]
        # the last piece starts at kb[-2] <= q0 and reaches q1 (it holds the diagonal)
        tiles.append((q0, q1, list(zip(kb[:-1], kb[1:]))))
    return tiles


@pytest.mark.parametrize("case", SPLITS, ids=[c[0] for c in SPLITS])
def test_random_key_pieces_merge_to_the_oracle(case):
    name, B, H, Hkv, T, d, S, dt = case
    x = _inputs(name, B, H, Hkv, T, d, S, dt)
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in NAMES}
    tiles = _random_tiling(T, seed=zlib.crc32(name.encode()))
    rng = np.random.default_rng(5)
    o_full = torch.empty_like(g["q"])
    lse_full = torch.empty(g["q"].shape[:3], dtype=torch.float32, device=dev)
    pieces_of = []
    for q0, q1, pieces in tiles:
        q = g["q"][:, :, q0:q1].contiguous()
        kd = g["kd"][:, :, q0:q1].contiguous() if S else None
        vd = g["vd"][:, :, q0:q1].contiguous() if S else None
        o_acc = torch.empty(q.shape, dtype=torch.float32, device=dev)
        lse_acc = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        order = rng.permutation(len(pieces))  # the merge order does not matter
        parts = []
        for n_merged, i in enumerate(order):
            k0, k1 = pieces[i]
            k = g["k"][:, :, k0:k1].contiguous()
            v = g["v"][:, :, k0:k1].contiguous()
            last = k1 == q1
            o_p, l_p = binding.moda_fwd_partial(q, k, v, kd if last else None, vd if last else None, q0 - k0)
            binding.moda_merge_partial(o_acc, lse_acc, o_p, l_p, first=n_merged == 0)
            parts.append((k0, k1, k, v, last))
        o_full[:, :, q0:q1] = binding.moda_convert_f32(o_acc, dt)
        lse_full[:, :, q0:q1] = lse_acc
        pieces_of.append((q0, q1, q, kd, vd, parts))
    torch.cuda.synchronize()
    hx = [host_view(x[n]) for n in NAMES]
    ro, rl = oracle.forward(*hx[:5])
    tol = TOL_OUT[dt]
    assert max_abs(as_f64(o_full), ro) < tol, max_abs(as_f64(o_full), ro)
    assert max_abs(as_f64(lse_full), rl) < tol, max_abs(as_f64(lse_full), rl)

    # backward of every pair, accumulated into whole-sequence float32 gradients
    dq = torch.zeros(g["q"].shape, dtype=torch.float32, device=dev)
    dk = torch.zeros(g["k"].shape, dtype=torch.float32, device=dev)
    dv = torch.zeros(g["v"].shape, dtype=torch.float32, device=dev)
    dkd = torch.zeros_like(g["kd"]) if S else None
    dvd = torch.zeros_like(g["vd"]) if S else None
    for q0, q1, q, kd, vd, parts in pieces_of:
        o = o_full[:, :, q0:q1].contiguous()
        lse = lse_full[:, :, q0:q1].contiguous()
        dout = g["dout"][:, :, q0:q1].contiguous()
        dq_acc = torch.zeros(q.shape, dtype=torch.float32, device=dev)
        for k0, k1, k, v, last in parts:
            dk_acc = torch.zeros(k.shape, dtype=torch.float32, device=dev)
            dv_acc = torch.zeros(k.shape, dtype=torch.float32, device=dev)
            _, _, _, pdkd, pdvd = binding.moda_bwd_partial(q, k, v, kd if last else None, vd if last else None, o,
                                                           lse, dout, q0 - k0, dq_acc, dk_acc, dv_acc)
            dk[:, :, k0:k1] += dk_acc
            dv[:, :, k0:k1] += dv_acc
            if last and S:
                dkd[:, :, q0:q1] = pdkd
                dvd[:, :, q0:q1] = pdvd
        dq[:, :, q0:q1] = dq_acc
    torch.cuda.synchronize()
    ref = oracle.backward(*hx)
    for nm, got, r in zip(("dq", "dk", "dv", "dkd", "dvd"), (dq, dk, dv, dkd, dvd), ref):
        if got is None:
            continue
        gg = as_f64(got)
        assert np.isfinite(gg).all(), nm
        assert rel_err(gg, r) < TOL_GRAD_REL, (nm, rel_err(gg, r))


def test_whole_sequence_partial_equals_moda_fwd_and_bwd_bitwise():
    """Tk = T, delta = 0 with the depth slots is moda_fwd's own problem: same kernels, same
    bits; the accumulating backward adds exactly moda_bwd's float32 values before rounding."""
    x = _inputs("whole", 1, 8, 2, 333, 64, 5, bf16)
    g = {n: x[n].cuda() for n in NAMES}
    o, lse = binding.moda_fwd(g["q"], g["k"], g["v"], g["kd"], g["vd"])
    o2, lse2 = binding.moda_fwd_partial(g["q"], g["k"], g["v"], g["kd"], g["vd"], 0)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    dq, dk, dv, dkd, dvd = binding.moda_bwd(g["q"], g["k"], g["v"], g["kd"], g["vd"], o, lse, g["dout"])
    acc = [torch.zeros(t.shape, dtype=torch.float32, device="cuda") for t in (g["q"], g["k"], g["v"])]
    _, _, _, dkd2, dvd2 = binding.moda_bwd_partial(g["q"], g["k"], g["v"], g["kd"], g["vd"], o, lse, g["dout"], 0,
                                                   *acc)
    torch.cuda.synchronize()
    for a, b in zip((dq, dk, dv), acc):
        assert torch.equal(a, binding.moda_convert_f32(b, bf16))
    assert torch.equal(dkd, dkd2) and torch.equal(dvd, dvd2)


def test_merge_edge_cases():
    dev = torch.device("cuda:0")
    B, H, T, d = 1, 2, 37, 128
    gen = torch.Generator().manual_seed(3)
    o_a = torch.randn(B, H, T, d, generator=gen).to(dev)
    l_a = torch.randn(B, H, T, generator=gen).to(dev)
    o_b = torch.randn(B, H, T, d, generator=gen).to(bf16).to(dev)
    l_b = torch.randn(B, H, T, generator=gen).to(dev)
    # first: the running state becomes the partial state, o_out its rounding
    acc, lacc = torch.full_like(o_a, float("nan")), torch.full_like(l_a, float("nan"))
    out = torch.empty(B, H, T, d, dtype=bf16, device=dev)
    binding.moda_merge_partial(acc, lacc, o_b, l_b, first=True, o_out=out)
    torch.cuda.synchronize()
    assert torch.equal(acc, o_b.float()) and torch.equal(lacc, l_b) and torch.equal(out, o_b)
    # a partial state without mass (lse = -inf) leaves the running state as it was
    acc, lacc = o_a.clone(), l_a.clone()
    binding.moda_merge_partial(acc, lacc, o_b, torch.full_like(l_b, float("-inf")))
    torch.cuda.synchronize()
    assert torch.equal(acc, o_a) and torch.equal(lacc, l_a)
    # two equal states merge to themselves, lse + ln 2
    acc, lacc = o_b.float().clone(), l_b.clone()
    binding.moda_merge_partial(acc, lacc, o_b, l_b)
    torch.cuda.synchronize()
    assert max_abs(acc.cpu().numpy(), o_b.float().cpu().numpy()) < 1e-5
    assert max_abs(lacc.cpu().numpy(), (l_b + np.log(2.0)).cpu().numpy()) < 1e-5


@pytest.mark.parametrize("n", [0, 1, 3, 4, 1027, 1 << 20])
def test_convert_rounds_like_round_to_nearest_even(n):
    gen = torch.Generator().manual_seed(n)
    src = (torch.randn(max(n, 1), generator=gen) * 100)[:n].cuda()
    out = binding.moda_convert_f32(src, bf16)
    out32 = binding.moda_convert_f32(src, f32)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), src.cpu().to(bf16))
    assert torch.equal(out32, src)


def test_ring_schedule_with_a_half_full_slot_ring():
    """A bounded slot buffer (capacity 8, 3 slots read, NaN in the unread ones) through the
    chunked path: the depth fold of each chunk reads only its first 3 slots."""
    B, H, Hkv, T, d, S, C = 1, 8, 2, 500, 64, 3, 8
    shape = Shape("cp_ring", B, H, Hkv, T, d, S, bf16, backward=True, slot_capacity=C)
    x = make_inputs(shape, seed=77)
    for n in ("kd", "vd"):
        x[n][:, :, :, S:] = float("nan")
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in NAMES}
    world, layout = 3, "contiguous"
    owned = cp.chunks_of(T, world, layout)
    loc = {n: [_split(g[n], owned[r]) for r in range(world)] for n in NAMES}
    kern = cp.LibraryKernels(slots=S)
    o, lse = cp.simulate_ring_forward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], T, world, layout,
                                      kernels=kern)
    grads = cp.simulate_ring_backward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], o, lse, loc["dout"], T,
                                      world, layout, kernels=kern)
    torch.cuda.synchronize()
    chunks = [c for cs in owned for c in cs]
    flat = lambda per_rank: [p for r in range(world) for p in per_rank[r]]  # noqa: E731
    hx = {n: host_view(x[n]) for n in NAMES}
    hx["kd"] = np.ascontiguousarray(hx["kd"][:, :, :, :S])
    hx["vd"] = np.ascontiguousarray(hx["vd"][:, :, :, :S])
    args = [hx[n] for n in NAMES]
    ro, rl = oracle.forward(*args[:5])
    assert max_abs(as_f64(_assemble(flat(o), chunks, T)), ro) < TOL_OUT[bf16]
    assert max_abs(as_f64(_assemble(flat(lse), chunks, T)), rl) < TOL_OUT[bf16]
    ref = oracle.backward(*args)
    for i, nm in enumerate(("dq", "dk", "dv")):
        got = as_f64(_assemble(flat(grads[i]), chunks, T))
        assert rel_err(got, ref[i]) < TOL_GRAD_REL, (nm, rel_err(got, ref[i]))
    for i, nm in ((3, "dkd"), (4, "dvd")):
        got = as_f64(_assemble(flat(grads[i]), chunks, T))
        assert np.all(got[:, :, :, S:] == 0), nm  # unread slots get zero gradient
        assert rel_err(got[:, :, :, :S], ref[i]) < TOL_GRAD_REL, (nm, rel_err(got[:, :, :, :S], ref[i]))
