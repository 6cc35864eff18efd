"""Helpers shared by the tests: device upload of seeded inputs and the parity metrics."""
from __future__ import annotations

import numpy as np
import torch

REL_L2_TOL = 1e-3   # relative L2 error bound of every floating-point output
MAX_ABS_TOL = 2e-3  # max-abs error bound of every floating-point output


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in inp.items()}


def rel_l2(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return float(num / den) if den > 0 else float(num)


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))


def assert_close(got, ref, what=""):
    r, m = rel_l2(got, ref), max_abs(got, ref)
    assert np.isfinite(np.asarray(got, np.float64)).all(), f"{what}: non-finite output"
    assert r <= REL_L2_TOL and m <= MAX_ABS_TOL, f"{what}: rel L2 {r:.3e} (<= {REL_L2_TOL}), max-abs {m:.3e} (<= {MAX_ABS_TOL})"
    return r, m
