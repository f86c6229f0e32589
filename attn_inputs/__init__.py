"""Seeded synthetic inputs for exact softmax attention.

This module is shared by the CPU oracle, the GPU tests and the benchmark. It
holds only random-number generation and the float32 -> bfloat16 storage
conversion (round to nearest, ties to even); none of the attention arithmetic
lives here.

Workload recipe (the attention microbenchmark of the FlashAttention-2 reading
note, papers.chlience.com, "结果 1"; and the "Evaluation Methodology" of the
paper-graph-ui summary, which says the kernels are timed on synthetic tensors):
Q, K, V and the upstream gradient dO are iid N(0, 1), drawn as float32 from
NumPy's PCG64 and rounded to bf16. Each tensor comes from its own child stream
of one SeedSequence, so every tensor is reproducible on its own and the bytes
are identical for the oracle and the GPU path.
"""

from __future__ import annotations

import numpy as np

# Base seed of the synthetic workloads; a config index is added to it.
BASE_SEED = 20230717

TENSORS = ("q", "k", "v", "do")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits.

    Inputs are finite by construction (normal draws, optionally multiplied by a
    power of two), so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def make_inputs(B: int, H: int, N: int, d: int, seed: int, *,
                peaked_frac: float = 0.0, peak_scale: float = 8.0,
                tensors=TENSORS) -> dict:
    """Return {name: uint16 array [B, H, N, d] of bf16 bits} for the named tensors.

    peaked_frac > 0 selects round(peaked_frac * N) query rows per (b, h),
    uniformly without replacement from a separate seeded stream, and multiplies
    those Q rows by peak_scale (a power of two, hence exact in bf16). This is
    the long-context stress input: rows whose logits have a much larger spread,
    so the running row maximum keeps moving late in the key loop.
    """
    if min(B, H, N, d) < 0:
        raise ValueError("negative size")
    children = np.random.SeedSequence(seed).spawn(len(TENSORS) + 1)
    out = {}
    shape = (B, H, N, d)
    for name, child in zip(TENSORS, children[:len(TENSORS)]):
        if name not in tensors:
            continue
        gen = np.random.Generator(np.random.PCG64(child))
        x = gen.standard_normal(size=shape, dtype=np.float32)
        if name == "q" and peaked_frac > 0.0 and N > 0:
            x = x.reshape(B * H, N, d)
            sel_gen = np.random.Generator(np.random.PCG64(children[-1]))
            n_peak = int(round(peaked_frac * N))
            for bh in range(B * H):
                rows = sel_gen.choice(N, size=n_peak, replace=False)
                x[bh, rows, :] *= np.float32(peak_scale)
            x = x.reshape(shape)
        out[name] = f32_to_bf16_bits(x).reshape(shape)
    return out


def peaked_rows(B: int, H: int, N: int, seed: int, peaked_frac: float) -> np.ndarray:
    """Row indices [B*H, n_peak] that make_inputs scales, for the same arguments."""
    children = np.random.SeedSequence(seed).spawn(len(TENSORS) + 1)
    sel_gen = np.random.Generator(np.random.PCG64(children[-1]))
    n_peak = int(round(peaked_frac * N))
    return np.stack([sel_gen.choice(N, size=n_peak, replace=False) for _ in range(B * H)]) \
        if B * H > 0 else np.zeros((0, n_peak), dtype=np.int64)


# The synthetic workloads, by name. Sizes follow the pages' benchmark shapes:
# hidden size 2048 split as d=64 x 32 heads or d=128 x 16 heads, 16k tokens per
# batch (B = 16384 / N), sequence lengths 512 .. 16k.
WORKLOADS = {
    "tiny_fwd": dict(B=1, H=1, N=128, d=64, causal=False, seed_index=0),
    "small_causal_fwdbwd": dict(B=2, H=4, N=1024, d=64, causal=True, seed_index=1),
    "long_causal_peaked": dict(B=1, H=16, N=32768, d=128, causal=True, seed_index=3, peaked_frac=0.01),
    "wide_head_d256": dict(B=1, H=2, N=16384, d=256, causal=False, seed_index=4),
}


def sweep_points():
    """The hidden-2048 sweep: (name, params) for every point."""
    pts = []
    for d, H in ((64, 32), (128, 16)):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            for causal in (False, True):
                B = 16384 // N
                name = f"sweep_d{d}_N{N}_{'causal' if causal else 'full'}"
                pts.append((name, dict(B=B, H=H, N=N, d=d, causal=causal, seed_index=2)))
    return pts


def seed_for(params: dict) -> int:
    return BASE_SEED + int(params.get("seed_index", 0))
