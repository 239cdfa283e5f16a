"""Context parallelism for MoDA: the positions 0..T-1 split over the ranks of a group.

Partitioning ("Mixture-of-Depths Attention", future work of frame "The main open cost
is retaining and reading depth history"):

* The positions are cut into chunks of (nearly) equal length.  ``contiguous`` gives rank
  r chunk r of ``world``; ``zigzag`` cuts ``2 * world`` chunks and gives rank r chunks r
  and 2 world - 1 - r, so every rank holds the same causal work.
* A rank keeps everything indexed by its own positions: q, o, lse, dout, dq, k, v, dk,
  dv and the depth slots kd, vd, dkd, dvd.  Depth slots are read only by their own
  position (frame "Depth retrieval is restricted to the same token position"), so the
  depth fold is the owner's: it enters the pair of a chunk with itself, and no depth byte
  crosses GPUs.
* Sequence K/V travel a ring: at step s rank r holds the K/V chunks of rank
  (r - s) mod world, sends them to rank r + 1 and receives the next from rank r - 1 while
  it computes.  A pair (query chunk, key chunk) is computed when the key chunk starts at
  or before the query chunk: the chunk with itself causally with its depth slots, an
  earlier chunk with every key visible.  Each pair is one ``fwd_partial`` call whose
  (O, lse) is merged into the rank's float32 running state by the online rule of frame
  "Shared online-softmax states preserve the joint operator".
* Backward: the same ring of K/V, plus float32 dK/dV accumulators that travel with them:
  each rank adds its queries' share of the visiting chunk's dK/dV and passes the
  accumulators on; one more hop after the last step returns them to their owner.  dQ and
  the depth gradients stay local.

Data moves with ``torch.distributed`` point-to-point operations (NCCL send/recv into
local device buffers on GPUs, gloo on CPU ranks); the compute of every pair runs in the
kernels behind ``kernels`` (the library's C ABI by default).  ``simulate_ring_forward``
and ``simulate_ring_backward`` run the same schedule for all ranks in one process, one
rank after the other (no kernel waits on another rank), for single-device checks.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Chunk:
    index: int   # global chunk index (chunks are ordered by position)
    start: int   # first position
    length: int  # positions


def chunks_of(T: int, world: int, layout: str = "contiguous"):
    """Per rank, the list of chunks it owns (ordered by position)."""
    if layout not in ("contiguous", "zigzag"):
        raise ValueError(f"unknown layout {layout!r}")
    n = world if layout == "contiguous" else 2 * world
    if world < 1 or T < n:
        raise ValueError(f"T={T} cannot be cut into {n} chunks")
    base, extra = divmod(T, n)
    chunks, start = [], 0
    for i in range(n):
        length = base + (1 if i < extra else 0)
        chunks.append(Chunk(i, start, length))
        start += length
    if layout == "contiguous":
        return [[chunks[r]] for r in range(world)]
    return [[chunks[r], chunks[n - 1 - r]] for r in range(world)]


def pair(qc: Chunk, kc: Chunk):
    """(Tk, delta, depth) of query chunk ``qc`` against key chunk ``kc``, or None when no key
    of ``kc`` is visible to ``qc`` (it starts after ``qc``)."""
    if kc.index > qc.index:
        return None
    if kc.index == qc.index:
        return kc.length, 0, True
    return kc.length, qc.start - kc.start, False


def owner_at(rank: int, step: int, world: int) -> int:
    """Rank whose K/V chunks rank ``rank`` holds at ring step ``step``."""
    return (rank - step) % world


def ring_pairs(rank: int, world: int, layout: str, T: int):
    """Per step, the pairs rank ``rank`` computes: (q sub-chunk, k sub-chunk, Tk, delta,
    depth), indices into its own and the visiting rank's chunk lists."""
    owned = chunks_of(T, world, layout)
    steps = []
    for s in range(world):
        kcs = owned[owner_at(rank, s, world)]
        todo = []
        for qi, qc in enumerate(owned[rank]):
            for ki, kc in enumerate(kcs):
                pr = pair(qc, kc)
                if pr is not None:
                    todo.append((qi, ki) + pr)
        steps.append(todo)
    return steps


# ---------------------------------------------------------------- kernels
class LibraryKernels:
    """The per-pair compute, through the library's C ABI (CUDA tensors)."""

    acc_dtype = torch.float32  # running states and gradient accumulators

    def __init__(self, scale=None, slots=None):
        from . import binding

        self.b = binding
        self.scale = scale
        self.slots = slots

    def fwd_partial(self, q, k, v, kd, vd, delta):
        return self.b.moda_fwd_partial(q, k, v, kd, vd, delta, scale=self.scale, slots=self.slots)

    def merge(self, o_acc, lse_acc, o_part, lse_part, first):
        self.b.moda_merge_partial(o_acc, lse_acc, o_part, lse_part, first=first)

    def bwd_partial(self, q, k, v, kd, vd, o, lse, dout, delta, dq_acc, dk_acc, dv_acc, dkd, dvd):
        self.b.moda_bwd_partial(q, k, v, kd, vd, o, lse, dout, delta, dq_acc, dk_acc, dv_acc, dkd, dvd,
                                scale=self.scale, slots=self.slots)

    def convert(self, src, dtype):
        return self.b.moda_convert_f32(src, dtype)


# ---------------------------------------------------------------- one step of one rank
def _forward_step(kernels, pairs, q, kd, vd, kv, state):
    """Computes and merges the pairs of one step; ``state`` = (o_acc, lse_acc, merged) lists
    per own chunk."""
    k, v = kv
    o_acc, lse_acc, merged = state
    for qi, ki, _tk, delta, depth in pairs:
        o_p, lse_p = kernels.fwd_partial(q[qi], k[ki], v[ki], kd[qi] if depth else None,
                                         vd[qi] if depth else None, delta)
        kernels.merge(o_acc[qi], lse_acc[qi], o_p, lse_p, first=not merged[qi])
        merged[qi] = True


def _backward_step(kernels, pairs, q, kd, vd, o, lse, dout, kv, dkv_acc, dq_acc, dkd, dvd):
    k, v = kv
    dk_acc, dv_acc = dkv_acc
    for qi, ki, _tk, delta, depth in pairs:
        kernels.bwd_partial(q[qi], k[ki], v[ki], kd[qi] if depth else None, vd[qi] if depth else None, o[qi],
                            lse[qi], dout[qi], delta, dq_acc[qi], dk_acc[ki], dv_acc[ki],
                            dkd[qi] if depth else None, dvd[qi] if depth else None)


def _new_state(q, acc_dtype):
    o_acc = [torch.empty(x.shape, dtype=acc_dtype, device=x.device) for x in q]
    lse_acc = [torch.empty(x.shape[:3], dtype=acc_dtype, device=x.device) for x in q]
    return o_acc, lse_acc, [False] * len(q)


def _kv_like(k, chunks):
    """Receive buffers for the K (or V) chunks ``chunks``, shaped like the local ones."""
    B, Hkv, _, d = k[0].shape
    return [torch.empty((B, Hkv, c.length, d), dtype=k[0].dtype, device=k[0].device) for c in chunks]


def _acc_like(k, chunks, acc_dtype):
    """Zeroed gradient accumulators for the K (or V) chunks ``chunks``."""
    B, Hkv, _, d = k[0].shape
    return [torch.zeros((B, Hkv, c.length, d), dtype=acc_dtype, device=k[0].device) for c in chunks]


# ---------------------------------------------------------------- the ring on a process group
class RingExchange:
    """Point-to-point ring transfers of lists of tensors: send to rank + 1, receive from
    rank - 1 (every rank posts its sends and receives in the same order)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def _global(self, r):
        return self.dist.get_global_rank(self.group, r) if self.group is not None else r

    def start(self, send, recv):
        nxt = self._global((self.rank + 1) % self.world)
        prv = self._global((self.rank - 1) % self.world)
        ops = [self.dist.P2POp(self.dist.isend, t, nxt, self.group) for t in send]
        ops += [self.dist.P2POp(self.dist.irecv, t, prv, self.group) for t in recv]
        return self.dist.batch_isend_irecv(ops) if ops else []

    @staticmethod
    def wait(reqs):
        for r in reqs:
            r.wait()


def ring_forward(q, k, v, kd, vd, T, layout="contiguous", group=None, kernels=None):
    """Context-parallel forward on this rank.  q, k, v, kd, vd: lists over this rank's
    chunks (``chunks_of(T, world, layout)[rank]``) of [B,H,len,d] / [B,Hkv,len,d] /
    [B,Hkv,len,C,d] tensors (kd, vd entries None without depth).  Returns (o, lse) lists
    for this rank's chunks, o in q's dtype and lse float32."""
    ex = RingExchange(group)
    kernels = kernels or LibraryKernels()
    owned = chunks_of(T, ex.world, layout)
    steps = ring_pairs(ex.rank, ex.world, layout, T)
    state = _new_state(q, kernels.acc_dtype)
    kv = (list(k), list(v))
    for s in range(ex.world):
        reqs, nxt = [], None
        if s + 1 < ex.world:
            src = owned[owner_at(ex.rank, s + 1, ex.world)]
            nxt = (_kv_like(k, src), _kv_like(v, src))
            reqs = ex.start(kv[0] + kv[1], nxt[0] + nxt[1])
        _forward_step(kernels, steps[s], q, kd, vd, kv, state)
        ex.wait(reqs)
        if nxt is not None:
            kv = nxt
    o_acc, lse_acc, _ = state
    return [kernels.convert(x, q[0].dtype) for x in o_acc], lse_acc


def ring_backward(q, k, v, kd, vd, o, lse, dout, T, layout="contiguous", group=None, kernels=None):
    """Context-parallel backward on this rank (lists over its chunks as for ring_forward; o,
    lse from ring_forward).  Returns (dq, dk, dv, dkd, dvd) lists in q's dtype (dkd, dvd
    entries None without depth)."""
    ex = RingExchange(group)
    kernels = kernels or LibraryKernels()
    owned = chunks_of(T, ex.world, layout)
    steps = ring_pairs(ex.rank, ex.world, layout, T)
    dq_acc = [torch.zeros(x.shape, dtype=kernels.acc_dtype, device=x.device) for x in q]
    dkd = [torch.empty_like(x) if x is not None else None for x in kd]
    dvd = [torch.empty_like(x) if x is not None else None for x in vd]
    kv = (list(k), list(v))
    acc = (_acc_like(k, owned[ex.rank], kernels.acc_dtype), _acc_like(k, owned[ex.rank], kernels.acc_dtype))
    for s in range(ex.world):
        reqs, nxt = [], None
        if s + 1 < ex.world:
            src = owned[owner_at(ex.rank, s + 1, ex.world)]
            nxt = (_kv_like(k, src), _kv_like(v, src))
            reqs = ex.start(kv[0] + kv[1], nxt[0] + nxt[1])
        _backward_step(kernels, steps[s], q, kd, vd, o, lse, dout, kv, acc, dq_acc, dkd, dvd)
        if ex.world > 1:
            # the accumulators of owner (rank - s) go on to rank + 1; after the last step
            # that is their owner
            src = owned[owner_at(ex.rank, s + 1, ex.world)]
            nacc = (_acc_like(k, src, kernels.acc_dtype), _acc_like(k, src, kernels.acc_dtype))
            ex.wait(ex.start(acc[0] + acc[1], nacc[0] + nacc[1]))
            acc = nacc
        ex.wait(reqs)
        if nxt is not None:
            kv = nxt
    dt = q[0].dtype
    return ([kernels.convert(x, dt) for x in dq_acc], [kernels.convert(x, dt) for x in acc[0]],
            [kernels.convert(x, dt) for x in acc[1]], dkd, dvd)


# ---------------------------------------------------------------- all ranks in one process
def simulate_ring_forward(q, k, v, kd, vd, T, world, layout="contiguous", kernels=None):
    """ring_forward for every rank in one process: q, k, v, kd, vd are per-rank lists of
    per-chunk lists.  Steps run rank after rank; the exchange is a rotation of references."""
    kernels = kernels or LibraryKernels()
    states = [_new_state(q[r], kernels.acc_dtype) for r in range(world)]
    for s in range(world):
        for r in range(world):
            src = owner_at(r, s, world)
            _forward_step(kernels, ring_pairs(r, world, layout, T)[s], q[r], kd[r], vd[r], (k[src], v[src]),
                          states[r])
    return ([[kernels.convert(x, q[r][0].dtype) for x in states[r][0]] for r in range(world)],
            [states[r][1] for r in range(world)])


def simulate_ring_backward(q, k, v, kd, vd, o, lse, dout, T, world, layout="contiguous", kernels=None):
    """ring_backward for every rank in one process (lists as for simulate_ring_forward)."""
    kernels = kernels or LibraryKernels()
    owned = chunks_of(T, world, layout)
    dq_acc = [[torch.zeros(x.shape, dtype=kernels.acc_dtype, device=x.device) for x in q[r]] for r in range(world)]
    dkd = [[torch.empty_like(x) if x is not None else None for x in kd[r]] for r in range(world)]
    dvd = [[torch.empty_like(x) if x is not None else None for x in vd[r]] for r in range(world)]
    acc = [(_acc_like(k[r], owned[r], kernels.acc_dtype), _acc_like(k[r], owned[r], kernels.acc_dtype))
           for r in range(world)]  # by owner
    for s in range(world):
        for r in range(world):
            src = owner_at(r, s, world)
            _backward_step(kernels, ring_pairs(r, world, layout, T)[s], q[r], kd[r], vd[r], o[r], lse[r], dout[r],
                           (k[src], v[src]), acc[src], dq_acc[r], dkd[r], dvd[r])
    dt = q[0][0].dtype
    return ([[kernels.convert(x, dt) for x in dq_acc[r]] for r in range(world)],
            [[kernels.convert(x, dt) for x in acc[r][0]] for r in range(world)],
            [[kernels.convert(x, dt) for x in acc[r][1]] for r in range(world)], dkd, dvd)
