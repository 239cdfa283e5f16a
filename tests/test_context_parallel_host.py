"""Host logic of the context-parallel T split, on CPU (no GPU).

* The partition: chunks cover 0..T-1 once, the ring visits every owner once per rank,
  and the pairs computed over all ranks and steps are exactly the causally visible
  (query chunk, key chunk) pairs, each once, the chunk-with-itself pairs carrying the
  depth slots.
* The ring exchange on two and three gloo ranks, with a float64 CPU stand-in for the four
  library calls: every rank receives the K/V chunks in the ring order, the dK/dV
  accumulators come home, and the assembled outputs and gradients equal the unchunked
  oracle.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from joint_sequence_depth_gb300 import context_parallel as cp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- partition and schedule
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("world,T", [(1, 5), (2, 37), (3, 100), (4, 64), (5, 11)])
def test_chunks_partition_the_positions(layout, world, T):
    if layout == "zigzag" and T < 2 * world:
        pytest.skip("too few positions")
    owned = cp.chunks_of(T, world, layout)
    assert len(owned) == world
    allc = sorted((c for cs in owned for c in cs), key=lambda c: c.index)
    assert [c.index for c in allc] == list(range(len(allc)))
    pos = 0
    for c in allc:
        assert c.start == pos and c.length >= 1
        pos += c.length
    assert pos == T
    lens = [c.length for c in allc]
    assert max(lens) - min(lens) <= 1


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 6])
def test_ring_computes_every_visible_pair_once(layout, world):
    T = 10 * world + 3
    owned = cp.chunks_of(T, world, layout)
    seen = []
    for r in range(world):
        owners = [cp.owner_at(r, s, world) for s in range(world)]
        assert sorted(owners) == list(range(world)) and owners[0] == r
        for s, pairs in enumerate(cp.ring_pairs(r, world, layout, T)):
            kcs = owned[owners[s]]
            for qi, ki, Tk, delta, depth in pairs:
                qc, kc = owned[r][qi], kcs[ki]
                assert kc.index <= qc.index
                assert Tk == kc.length and delta == qc.start - kc.start
                assert depth == (kc.index == qc.index)
                # the chunk geometry moda_fwd_partial accepts
                assert delta >= 0 and 1 <= Tk <= qc.length + delta
                seen.append((qc.index, kc.index))
    n = len([c for cs in owned for c in cs])
    assert sorted(seen) == sorted((i, j) for i in range(n) for j in range(i + 1))


def test_zigzag_balances_the_causal_work():
    world, T = 4, 4096
    work = []
    for r in range(world):
        owned = cp.chunks_of(T, world, "zigzag")
        w = 0
        for s, pairs in enumerate(cp.ring_pairs(r, world, "zigzag", T)):
            for qi, ki, Tk, delta, depth in pairs:
                Tq = owned[r][qi].length
                # visible (query, key) products of the pair
                w += sum(min(Tk, t + delta + 1) for t in range(Tq))
        work.append(w)
    assert max(work) / min(work) < 1.01
    contiguous = []
    for r in range(world):
        owned = cp.chunks_of(T, world, "contiguous")
        contiguous.append(sum(sum(min(Tk, t + delta + 1) for t in range(owned[r][qi].length))
                              for pairs in cp.ring_pairs(r, world, "contiguous", T) for qi, _, Tk, delta, _ in pairs))
    assert max(contiguous) / min(contiguous) > 5


# ---------------------------------------------------------------- float64 stand-in kernels
class CpuKernels:
    """float64 CPU stand-in of moda_fwd_partial / moda_merge_partial / moda_bwd_partial /
    moda_convert_f32, so the exchange can run on gloo ranks.  It records, per call, which
    key chunk arrived (found by comparing against the full K)."""

    acc_dtype = torch.float64

    def __init__(self, scale, k_full=None):
        self.scale = scale
        self.k_full = k_full
        self.seen = []

    def _which(self, k):
        if self.k_full is None:
            return None
        Tk = k.shape[2]
        for start in range(self.k_full.shape[2] - Tk + 1):
            if torch.equal(self.k_full[:, :, start:start + Tk], k):
                return start
        return -1

    def _scores(self, q, k, kd, delta):
        G = q.shape[1] // k.shape[1]
        kk = k.repeat_interleave(G, dim=1)
        s = self.scale * q @ kk.transpose(-1, -2)
        t = torch.arange(q.shape[2])[:, None]
        j = torch.arange(k.shape[2])[None, :]
        s = s.masked_fill(j > t + delta, float("-inf"))
        sd = None
        if kd is not None:
            sd = self.scale * torch.einsum("bhtd,bhtsd->bhts", q, kd.repeat_interleave(G, dim=1))
        return s, sd, G

    def fwd_partial(self, q, k, v, kd, vd, delta):
        self.seen.append(self._which(k))
        s, sd, G = self._scores(q, k, kd, delta)
        allw = s if sd is None else torch.cat([s, sd], dim=-1)
        lse = torch.logsumexp(allw, dim=-1)
        o = torch.exp(s - lse[..., None]) @ v.repeat_interleave(G, dim=1)
        if sd is not None:
            o = o + torch.einsum("bhts,bhtsd->bhtd", torch.exp(sd - lse[..., None]), vd.repeat_interleave(G, dim=1))
        return o, lse

    def merge(self, o_acc, lse_acc, o_part, lse_part, first):
        if first:
            o_acc.copy_(o_part)
            lse_acc.copy_(lse_part)
            return
        m = torch.maximum(lse_acc, lse_part)
        wa, wb = torch.exp(lse_acc - m), torch.exp(lse_part - m)
        o_acc.copy_((wa[..., None] * o_acc + wb[..., None] * o_part) / (wa + wb)[..., None])
        lse_acc.copy_(m + torch.log(wa + wb))

    def bwd_partial(self, q, k, v, kd, vd, o, lse, dout, delta, dq_acc, dk_acc, dv_acc, dkd, dvd):
        s, sd, G = self._scores(q, k, kd, delta)
        B, Hkv, Tk, d = k.shape
        D = (dout * o).sum(-1, keepdim=True)
        p = torch.exp(s - lse[..., None])
        ds = p * (dout @ v.repeat_interleave(G, dim=1).transpose(-1, -2) - D)
        dq_acc += self.scale * ds @ k.repeat_interleave(G, dim=1)
        dk_acc += (self.scale * ds.transpose(-1, -2) @ q).reshape(B, Hkv, G, Tk, d).sum(2)
        dv_acc += (p.transpose(-1, -2) @ dout).reshape(B, Hkv, G, Tk, d).sum(2)
        if sd is not None:
            T, S = q.shape[2], kd.shape[3]
            pd = torch.exp(sd - lse[..., None])
            dsd = pd * (torch.einsum("bhtd,bhtsd->bhts", dout, vd.repeat_interleave(G, dim=1)) - D)
            dq_acc += self.scale * torch.einsum("bhts,bhtsd->bhtd", dsd, kd.repeat_interleave(G, dim=1))
            dkd.copy_((self.scale * torch.einsum("bhts,bhtd->bhtsd", dsd, q)).reshape(B, Hkv, G, T, S, d).sum(2))
            dvd.copy_(torch.einsum("bhts,bhtd->bhtsd", pd, dout).reshape(B, Hkv, G, T, S, d).sum(2))

    def convert(self, src, dtype):
        return src.to(dtype)


def _problem(seed, B=1, H=4, Hkv=2, T=37, S=3, d=16):
    g = np.random.default_rng(seed)
    x = {n: g.standard_normal(shape) for n, shape in (
        ("q", (B, H, T, d)), ("k", (B, Hkv, T, d)), ("v", (B, Hkv, T, d)), ("kd", (B, Hkv, T, S, d)),
        ("vd", (B, Hkv, T, S, d)), ("dout", (B, H, T, d)))}
    return x, 1.0 / np.sqrt(d)


def _split(t, chunks, dim=2):
    return [t.narrow(dim, c.start, c.length).contiguous() for c in chunks]


def _assemble(parts, chunks, T, dim=2):
    shape = list(parts[0].shape)
    shape[dim] = T
    out = torch.empty(shape, dtype=parts[0].dtype)
    for p, c in zip(parts, chunks):
        out.narrow(dim, c.start, c.length).copy_(p)
    return out


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, layout, results):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, scale = _problem(seed=7)
        t = {n: torch.from_numpy(a) for n, a in x.items()}
        T = t["q"].shape[2]
        mine = cp.chunks_of(T, world, layout)[rank]
        loc = {n: _split(a, mine) for n, a in t.items()}
        kern = CpuKernels(scale, k_full=t["k"])
        o, lse = cp.ring_forward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], T, layout, kernels=kern)
        fwd_seen = list(kern.seen)
        grads = cp.ring_backward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], o, lse, loc["dout"], T, layout,
                                 kernels=kern)
        results[rank] = (o, lse, grads, fwd_seen)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,layout", [(2, "contiguous"), (3, "contiguous"), (2, "zigzag")])
def test_ring_exchange_on_gloo_ranks_matches_the_oracle(world, layout):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, layout, results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    assert sorted(res) == list(range(world))
    x, scale = _problem(seed=7)
    T = x["q"].shape[2]
    owned = cp.chunks_of(T, world, layout)
    # exchange order: rank r's forward calls saw the key chunks of owners r, r-1, ... in ring order
    for r in range(world):
        expect = []
        for s, pairs in enumerate(cp.ring_pairs(r, world, layout, T)):
            kcs = owned[cp.owner_at(r, s, world)]
            expect += [kcs[ki].start for _, ki, *_ in pairs]
        assert res[r][3] == expect, (r, res[r][3], expect)
    chunks = [c for cs in owned for c in cs]
    o = _assemble([p for r in range(world) for p in res[r][0]], chunks, T)
    lse = _assemble([p for r in range(world) for p in res[r][1]], chunks, T)
    ro, rl = oracle.forward(x["q"], x["k"], x["v"], x["kd"], x["vd"], scale=scale)
    assert np.max(np.abs(o.numpy() - ro)) < 1e-10
    assert np.max(np.abs(lse.numpy() - rl)) < 1e-10
    ref = oracle.backward(x["q"], x["k"], x["v"], x["kd"], x["vd"], x["dout"], scale=scale)
    for i, name in enumerate(("dq", "dk", "dv", "dkd", "dvd")):
        got = _assemble([p for r in range(world) for p in res[r][2][i]], chunks, T)
        assert np.max(np.abs(got.numpy() - ref[i])) < 1e-10, name


def test_simulated_ring_equals_the_oracle_on_cpu():
    """The single-process simulation (used by the GPU tests) with the same stand-in."""
    x, scale = _problem(seed=11, T=50)
    t = {n: torch.from_numpy(a) for n, a in x.items()}
    T = 50
    for world, layout in ((3, "contiguous"), (3, "zigzag"), (1, "contiguous")):
        owned = cp.chunks_of(T, world, layout)
        loc = {n: [_split(a, owned[r]) for r in range(world)] for n, a in t.items()}
        kern = CpuKernels(scale)
        o, lse = cp.simulate_ring_forward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], T, world, layout,
                                          kernels=kern)
        grads = cp.simulate_ring_backward(loc["q"], loc["k"], loc["v"], loc["kd"], loc["vd"], o, lse, loc["dout"], T,
                                          world, layout, kernels=kern)
        chunks = [c for cs in owned for c in cs]
        flat = lambda per_rank: [p for r in range(world) for p in per_rank[r]]  # noqa: E731
        ro, rl = oracle.forward(x["q"], x["k"], x["v"], x["kd"], x["vd"], scale=scale)
        assert np.max(np.abs(_assemble(flat(o), chunks, T).numpy() - ro)) < 1e-10
        ref = oracle.backward(x["q"], x["k"], x["v"], x["kd"], x["vd"], x["dout"], scale=scale)
        for i in range(5):
            assert np.max(np.abs(_assemble(flat(grads[i]), chunks, T).numpy() - ref[i])) < 1e-10
