"""Seeded synthetic inputs for MoDA, shared by the tests, the smoke check and the benchmark.

This module holds no MoDA arithmetic: it only names the workload shapes and
draws i.i.d. N(0, 1) tensors from a seeded ``torch.Generator``, in a fixed
order (q, k, v, kd, vd, then dout), in float32, then rounds them to the storage
type (bf16 round-to-nearest-even).  The kernel benchmark on the MoDA page
(Table 2 / Table 7) times random tensors, so these synthetic inputs are the
workload itself, not a stand-in for a dataset.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    """One MoDA problem: B batch, H query heads, Hkv kv heads, T tokens, d head dim,
    S depth slots per position (the depth slots of the layer's history H_l)."""

    name: str
    B: int
    H: int
    Hkv: int
    T: int
    d: int
    S: int
    dtype: torch.dtype
    backward: bool = False
    # bounded slot buffer: slots per position in kd/vd memory (0: exactly S); the first S
    # are read, the rest stand for slots a ring has not filled yet
    slot_capacity: int = 0

    @property
    def S_mem(self) -> int:
        return self.slot_capacity if self.slot_capacity > 0 else self.S

    @property
    def G(self) -> int:
        return self.H // self.Hkv

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.dtype == torch.bfloat16 else "f32"


# The workloads MoDA is measured and checked on.
WORKLOADS = {
    "fp32_small": Shape("fp32_small", 1, 2, 2, 256, 64, 4, torch.float32),
    "bf16_mha": Shape("bf16_mha", 2, 16, 16, 2048, 128, 8, torch.bfloat16),
    "bf16_gqa": Shape("bf16_gqa", 4, 32, 8, 4096, 128, 24, torch.bfloat16),
    "bf16_long": Shape("bf16_long", 1, 32, 8, 16384, 128, 48, torch.bfloat16),
    "bf16_train": Shape("bf16_train", 8, 16, 4, 4096, 64, 32, torch.bfloat16, backward=True),
    # a quarter of the training batch: the size kernel profiles are captured on
    "bf16_train_quarter": Shape("bf16_train_quarter", 2, 16, 4, 4096, 64, 32, torch.bfloat16, backward=True),
    # the training step while a 32-slot ring is half full: 16 slots read of 32 in memory
    "bf16_train_ring_half": Shape("bf16_train_ring_half", 8, 16, 4, 4096, 64, 16, torch.bfloat16, backward=True,
                                  slot_capacity=32),
}

# seed of each workload (its index in the list above, from 1)
SEEDS = {name: i + 1 for i, name in enumerate(WORKLOADS)}


def make_inputs(shape: Shape, seed: int, device="cpu", with_dout: bool | None = None, dtype=None):
    """Draw q, k, v, kd, vd (and dout when requested) for ``shape``.

    Layouts: q/dout [B,H,T,d]; k/v [B,Hkv,T,d]; kd/vd [B,Hkv,T,S,d]; all dense
    row-major.  The generator lives on ``device`` (CPU and CUDA streams differ,
    so a given use always draws on the same device).
    """
    dtype = dtype or shape.dtype
    if with_dout is None:
        with_dout = shape.backward
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B, H, Hkv, T, d, S = shape.B, shape.H, shape.Hkv, shape.T, shape.d, shape.S
    dims = {
        "q": (B, H, T, d),
        "k": (B, Hkv, T, d),
        "v": (B, Hkv, T, d),
        "kd": (B, Hkv, T, shape.S_mem, d),
        "vd": (B, Hkv, T, shape.S_mem, d),
    }
    if with_dout:
        dims["dout"] = (B, H, T, d)
    out = {}
    for key, shp in dims.items():
        x = torch.randn(shp, generator=gen, device=device, dtype=torch.float32)
        out[key] = x if dtype == torch.float32 else x.to(dtype)
        del x
    return out


def scaled(shape: Shape, **changes) -> Shape:
    """A copy of ``shape`` with some sizes changed (for small parity cases)."""
    fields = dict(shape.__dict__)
    fields.update(changes)
    return Shape(**fields)


# Decode steps: one new token per sequence over a cache of T positions (its own included).
# Shape.T is the number of cached positions; Shape.S the depth slots of the new position.
DECODE_WORKLOADS = {
    "bf16_decode_gqa": Shape("bf16_decode_gqa", 8, 32, 8, 32768, 128, 48, torch.bfloat16),
    "bf16_decode_mha": Shape("bf16_decode_mha", 4, 32, 32, 16384, 128, 8, torch.bfloat16),
    "bf16_decode_d64": Shape("bf16_decode_d64", 16, 16, 4, 32768, 64, 32, torch.bfloat16),
}
DECODE_SEEDS = {name: 101 + i for i, name in enumerate(DECODE_WORKLOADS)}


def make_decode_inputs(shape: Shape, seed: int, device="cpu", capacity: int | None = None):
    """Draw a decode step's q [B,H,d], k/v cache [B,Hkv,capacity,d] (capacity >= T; the
    positions past T are drawn too and must not influence the step) and kd/vd [B,Hkv,S,d],
    i.i.d. N(0, 1) in float32 in that order, rounded to the storage type."""
    cap = capacity or shape.T
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B, H, Hkv, d, S = shape.B, shape.H, shape.Hkv, shape.d, shape.S
    dims = {"q": (B, H, d), "k": (B, Hkv, cap, d), "v": (B, Hkv, cap, d), "kd": (B, Hkv, S, d), "vd": (B, Hkv, S, d)}
    out = {}
    for key, shp in dims.items():
        x = torch.randn(shp, generator=gen, device=device, dtype=torch.float32)
        out[key] = x if shape.dtype == torch.float32 else x.to(shape.dtype)
        del x
    return out


# Depth-KV writes: one layer's contributions to the depth cache of a workload above.
# The model width is H * d (the query heads side by side); the projection weights map it
# to the Hkv * d columns of the depth keys (values).
WRITE_WORKLOADS = {
    "bf16_write_train": scaled(WORKLOADS["bf16_train"], name="bf16_write_train", backward=False),
    "bf16_write_gqa": scaled(WORKLOADS["bf16_gqa"], name="bf16_write_gqa"),
}
WRITE_SEEDS = {name: 201 + i for i, name in enumerate(WRITE_WORKLOADS)}


def d_model(shape: Shape) -> int:
    return shape.H * shape.d


def make_write_inputs(shape: Shape, seed: int, device="cpu", Dm: int | None = None):
    """Draw k, v [B,Hkv,T,d], kd, vd [B,Hkv,T,S,d], x [B,T,Dm] (Dm defaults to H*d) and
    wk, wv [Dm, Hkv*d], in that order, i.i.d. N(0, 1) in float32; the weights are then
    divided by sqrt(Dm) so that projected values have unit variance like the rest; all
    are rounded to the storage type."""
    Dm = Dm or d_model(shape)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B, Hkv, T, d, S = shape.B, shape.Hkv, shape.T, shape.d, shape.S
    dims = {"k": (B, Hkv, T, d), "v": (B, Hkv, T, d), "kd": (B, Hkv, T, S, d), "vd": (B, Hkv, T, S, d),
            "x": (B, T, Dm), "wk": (Dm, Hkv * d), "wv": (Dm, Hkv * d)}
    out = {}
    for key, shp in dims.items():
        x = torch.randn(shp, generator=gen, device=device, dtype=torch.float32)
        if key in ("wk", "wv"):
            x = x / float(Dm) ** 0.5
        out[key] = x if shape.dtype == torch.float32 else x.to(shape.dtype)
        del x
    return out
