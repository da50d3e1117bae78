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


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (the largest rounding error
    of an exact value stored as bf16)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


# Output tolerances (the attention output is bf16).  The max bound applies to
# the kernel's error beyond the rounding every bf16 output of the exact value
# carries (half a bf16 ulp at |exact|); the mean bound applies to the raw
# difference from the fp64 oracle.
MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3


def output_errors(got: np.ndarray, exact: np.ndarray):
    """(max excess over half an ulp, mean raw, max raw) of got vs exact."""
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    raw = np.abs(got - exact)
    if raw.size == 0:
        return 0.0, 0.0, 0.0
    excess = np.maximum(raw - bf16_half_ulp(exact), 0.0)
    return float(excess.max()), float(raw.mean()), float(raw.max())


def assert_close(got, exact, what=""):
    mx, mean, raw = output_errors(got, exact)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, \
        f"{what}: max err beyond bf16 rounding {mx:.3g} (tol {MAX_ABS_TOL}), mean abs {mean:.3g} " \
        f"(tol {MEAN_ABS_TOL}), raw max {raw:.3g}"
    return mx, mean
