"""Helpers shared by the GPU parity tests (host-side only)."""

from __future__ import annotations

import numpy as np

from attn_inputs import make_inputs, bf16_bits_to_f64

# Tolerances of the parity bar: O absolute 1e-2, L absolute 2e-3, gradients
# max|err| / max|ref| <= 2e-2 per tensor, all against the float64 oracle on
# the same bf16 inputs.
TOL_O = 1e-2
TOL_LSE = 2e-3
TOL_GRAD_REL = 2e-2


def to_device(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_host64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def scale_f32(d: int) -> float:
    """The softmax scale as the float32 value the library receives."""
    return float(np.float32(1.0 / np.sqrt(d)))


def inputs(B, H, N, d, seed, **kw):
    x = make_inputs(B, H, N, d, seed, **kw)
    return x, {k: bf16_bits_to_f64(v) for k, v in x.items()}


def sampled_pairs(B: int, H: int, seed: int, n_random: int = 2):
    """(0,0), (B-1,H-1) and n_random seeded random (b,h) pairs, deduplicated."""
    rng = np.random.default_rng(seed)
    pairs = [(0, 0), (B - 1, H - 1)]
    for _ in range(n_random):
        pairs.append((int(rng.integers(B)), int(rng.integers(H))))
    out = []
    for p in pairs:
        if p not in out:
            out.append(p)
    return out


def sampled_rows(N: int, seed: int, n: int = 512):
    """First and last 128 rows plus n seeded random rows (sorted, unique)."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(128, N))) | set(range(max(0, N - 128), N))
    rows |= set(int(r) for r in rng.choice(N, size=min(n, N), replace=False))
    return np.array(sorted(rows))
