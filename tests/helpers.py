"""Shared test helpers: run the oracle on a workload, compare outputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def pool_bytes(pool: torch.Tensor) -> np.ndarray:
    return pool.contiguous().view(torch.uint8).cpu().numpy().reshape(-1).copy()


def run_oracle(w, queries, keys, values, pool_before, sink=None, nthreads=0):
    """Oracle forward on a CPU copy of the pool: (out fp64, pool bytes after)."""
    p = oracle.make_params(**w.params())
    cache = pool_bytes(pool_before)
    out, cache = oracle.forward(p, queries, keys, values, cache, w.kv_lens,
                                w.block_tables, w.query_start_loc, w.num_seqs,
                                None if sink is None else sink.numpy(), nthreads)
    return out, cache


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even), back as fp64."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


# Output tolerances: the kernel's bf16 output against the oracle's exact value
# rounded to bf16 (the interface's output dtype).
MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3


def output_errors(got: np.ndarray, exact: np.ndarray):
    """(max abs, mean abs) of got - bf16(exact), and max abs of got - exact."""
    got = np.asarray(got, np.float64)
    ref = bf16_round(exact)
    d = np.abs(got - ref)
    raw = np.abs(got - exact)
    if d.size == 0:
        return 0.0, 0.0, 0.0
    return float(d.max()), float(d.mean()), float(raw.max())


def assert_close(got, exact, what=""):
    mx, mean, raw = output_errors(got, exact)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, \
        f"{what}: max abs {mx:.3g} (tol {MAX_ABS_TOL}), mean abs {mean:.3g} (tol {MEAN_ABS_TOL}), raw max {raw:.3g}"
    return mx, mean
