"""Seeded synthetic inputs for a QSA layer (random draws only, no attention arithmetic).

This module is the one piece shared by the CUDA path's callers and the CPU oracle's
callers: both receive the same arrays from here.  It holds only random number draws and
array shapes, never a step of the method.

Workload shapes follow the layer the pages measure ("round 6 track b - qsa flash",
actual runs; "opus_r9_qsa", result table): 2 KV groups x 12 query heads per group, head
dim 256, one fp16 scale per 64 elements of a K or V row, rng seed 5 (+ layer index).

Distributions:
  q    : standard normal, rounded to fp16                      [T][24][256]
  kq,vq: int8 codes uniform in [-127, 127]                     [n_cells][2][256]
  ksc,vsc: uniform in [0.005, 0.02], rounded to fp16           [n_cells][2][4]
"""
from __future__ import annotations

import numpy as np

N_GROUPS = 2
HEADS_PER_GROUP = 12
N_HEADS = N_GROUPS * HEADS_PER_GROUP
HEAD_DIM = 256
SCALE_BLOCK = 64
N_BLOCKS = HEAD_DIM // SCALE_BLOCK
PART_STRIDE = HEAD_DIM + 2  # o[256], m, l per (chunk, head)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def layer_inputs(T: int, n_cells: int, seed: int = 5) -> dict:
    """Queries for T new tokens and an n_cells-cell int8 KV cache with fp16 scales."""
    rng = _rng(seed)
    q = rng.standard_normal((T, N_HEADS, HEAD_DIM), dtype=np.float32).astype(np.float16)
    kq = rng.integers(-127, 128, size=(n_cells, N_GROUPS, HEAD_DIM), dtype=np.int8)
    vq = rng.integers(-127, 128, size=(n_cells, N_GROUPS, HEAD_DIM), dtype=np.int8)
    ksc = rng.uniform(0.005, 0.02, size=(n_cells, N_GROUPS, N_BLOCKS)).astype(np.float16)
    vsc = rng.uniform(0.005, 0.02, size=(n_cells, N_GROUPS, N_BLOCKS)).astype(np.float16)
    return {"q": q, "kq": kq, "vq": vq, "ksc": ksc, "vsc": vsc}


def fp16_rows(n_cells: int, seed: int = 5, spread: float = 1.0) -> np.ndarray:
    """fp16 K or V rows [n_cells][2][256] to be quantised (normal, per-row random gain)."""
    rng = _rng(seed)
    gain = np.exp(rng.uniform(-2.0, 2.0, size=(n_cells, N_GROUPS, 1))) * spread
    x = rng.standard_normal((n_cells, N_GROUPS, HEAD_DIM)) * gain
    return x.astype(np.float16)


def merge_partials(n_chunks, chunk_cap: int, seed: int = 5) -> np.ndarray:
    """Random split-KV partials [N][chunk_cap][24][258] fp32 for merge-only tests.

    o is drawn as l * (a point in [-1, 1]), m is normal with spread 3 (so chunks differ by
    many e-folds), l in [1, 64].  Slots at or beyond a token's chunk count are NaN so a
    merge that reads them is caught.
    """
    rng = _rng(seed)
    n_chunks = np.asarray(n_chunks, dtype=np.int32)
    N = len(n_chunks)
    part = np.full((N, chunk_cap, N_HEADS, PART_STRIDE), np.nan, dtype=np.float32)
    for t in range(N):
        c = int(n_chunks[t])
        l = rng.uniform(1.0, 64.0, size=(c, N_HEADS)).astype(np.float32)
        m = (rng.standard_normal((c, N_HEADS)) * 3.0).astype(np.float32)
        o = (rng.uniform(-1.0, 1.0, size=(c, N_HEADS, HEAD_DIM)) * l[..., None]).astype(np.float32)
        part[t, :c, :, :HEAD_DIM] = o
        part[t, :c, :, HEAD_DIM] = m
        part[t, :c, :, HEAD_DIM + 1] = l
    return part


def gate_input(T: int, seed: int = 5, spread: float = 2.0) -> np.ndarray:
    """Output-gate values [T][24][256] fp16, normal with standard deviation `spread` (a mix of
    nearly closed, half open and nearly open gates)."""
    rng = _rng(seed)
    return (rng.standard_normal((T, N_HEADS, HEAD_DIM)) * spread).astype(np.float16)


def prep_inputs(T: int, seed: int = 5) -> dict:
    """Raw projections of T new tokens for the fused prep: q_raw [T][24][256], k_raw and v_raw
    [T][2][256] fp16 (normal with a random gain per row), and the RMS-norm gains q_gamma,
    k_gamma [256] fp32 (1 + 0.1 N(0,1))."""
    rng = _rng(seed)
    def rows(shape):
        gain = np.exp(rng.uniform(-1.0, 1.0, size=shape[:-1] + (1,)))
        return (rng.standard_normal(shape) * gain).astype(np.float16)
    return {"q_raw": rows((T, N_HEADS, HEAD_DIM)), "k_raw": rows((T, N_GROUPS, HEAD_DIM)),
            "v_raw": rows((T, N_GROUPS, HEAD_DIM)),
            "q_gamma": (1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32),
            "k_gamma": (1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32)}
