"""Helpers shared by the GPU parity tests: host copies for the oracle and error measures."""
import numpy as np
import torch

# Tolerances against the float64 oracle: max-abs for outputs (fp32 / bf16 inputs)
# and max|g - g_ref| / max|g_ref| per gradient tensor.
TOL_OUT = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
TOL_GRAD_REL = 3e-2


def host_view(t: torch.Tensor) -> np.ndarray:
    """numpy view of a CPU tensor in the oracle's storage convention (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def rel_err(g, ref) -> float:
    g = np.asarray(g, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def sample_rows(shape, n, seed):
    """Flat row indices (b*H+h)*T+t: tile edges, the last position, and random rows."""
    rng = np.random.default_rng(seed)
    B, H, T = shape.B, shape.H, shape.T
    ts = sorted({0, 1, min(T - 1, 63), min(T - 1, 64), min(T - 1, 127), min(T - 1, 128), T // 2, T - 2, T - 1})
    rows = []
    for t in ts:
        b, h = rng.integers(B), rng.integers(H)
        rows.append((b * H + h) * T + t)
    rows += list(rng.integers(0, B * H * T, size=n))
    return np.unique(np.array(rows, dtype=np.int64))


def sample_positions(shape, n, seed):
    """Flat positions (b*Hkv+g)*T+t for the backward's position part."""
    rng = np.random.default_rng(seed)
    B, Hkv, T = shape.B, shape.Hkv, shape.T
    pos = [(rng.integers(B) * Hkv + rng.integers(Hkv)) * T + t for t in (0, T - 1, min(T - 1, 128))]
    pos += list(rng.integers(0, B * Hkv * T, size=n))
    return np.unique(np.array(pos, dtype=np.int64))


def sample_keys(shape, n, seed):
    """Flat sequence keys (b*Hkv+g)*T+j from three (b, kv head) pairs: the last keys (short
    sums), the first keys j < 128 (the longest dK/dV sums, from the longest-running dK/dV
    work), keys around the 128-key tile edges and random keys over the whole range."""
    rng = np.random.default_rng(seed)
    B, Hkv, T = shape.B, shape.Hkv, shape.T
    pairs = {(int(rng.integers(B)), int(rng.integers(Hkv))) for _ in range(3)}
    ks = []
    for b, g in sorted(pairs):
        base = (b * Hkv + g) * T
        js = {T - 1, T - 2, max(0, T - 130), 0, 1, min(T - 1, 127), min(T - 1, 128)}
        js |= {int(j) for j in rng.integers(0, min(T, 128), size=2)}
        js |= {int(j) for j in rng.integers(0, T, size=max(1, n // len(pairs)))}
        ks += [base + j for j in js]
    return np.unique(np.array(ks, dtype=np.int64))
