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


# Output tolerances (the attention output is bf16), as stated for this op:
# max |got - exact| <= 1e-2 and mean |got - exact| <= 1e-3 against the fp64
# oracle.  The max bound is taken literally wherever it can be met, that is
# wherever |exact| < 4: there half a bf16 ulp is at most 2^-7 ~ 0.0078, so
# even the correctly rounded output lies within it.  From |exact| >= 4 on,
# half an ulp (>= 2^-6 = 0.0156) alone exceeds 1e-2, so there the bound
# allows the output's own rounding on top: |got - exact| <= ulp/2 + 1e-2.
MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3
ROUNDING_FLOOR = 4.0  # |exact| from which the bf16 rounding alone exceeds MAX_ABS_TOL


def max_abs_bound(exact: np.ndarray) -> np.ndarray:
    """Per-element bound on |got - exact|: 1e-2 below |exact| = 4, half a
    bf16 ulp of exact plus 1e-2 from there on."""
    exact = np.asarray(exact, np.float64)
    return np.where(np.abs(exact) < ROUNDING_FLOOR, MAX_ABS_TOL,
                    bf16_half_ulp(exact) + MAX_ABS_TOL)


def output_errors(got: np.ndarray, exact: np.ndarray):
    """(worst ratio of |got - exact| to its bound, mean raw, max raw)."""
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    raw = np.abs(got - exact)
    if raw.size == 0:
        return 0.0, 0.0, 0.0
    return float((raw / max_abs_bound(exact)).max()), float(raw.mean()), float(raw.max())


def assert_close(got, exact, what=""):
    """Asserts the stated bounds; returns (max raw error, mean raw error)."""
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    ratio, mean, raw = output_errors(got, exact)
    where = ""
    if ratio > 1.0:
        r = np.abs(got - exact) / max_abs_bound(exact)
        i = np.unravel_index(int(np.argmax(r)), r.shape)
        where = f"; worst at index {tuple(int(x) for x in i)}: got {got[i]:.6g}, exact {exact[i]:.6g}"
    assert ratio <= 1.0 and mean <= MEAN_ABS_TOL, \
        f"{what}: max abs err {raw:.4g} (bound 1e-2 below |exact| 4, ulp/2 + 1e-2 above; " \
        f"worst ratio {ratio:.3g}), mean abs err {mean:.3g} (tol {MEAN_ABS_TOL}){where}"
    return raw, mean


# Non-finite bit patterns for the slots of a pool that no query may read:
# bf16 quiet NaN, +Inf, -Inf and a negative NaN with a payload; e4m3 (fn)
# has no infinities, its NaN codes are 0x7F and 0xFF.
NONFINITE_BF16 = (0x7FC0, 0x7F80, 0xFF80, 0xFFC1)
NONFINITE_E4M3 = (0x7F, 0xFF)


def read_slots(w) -> np.ndarray:
    """Boolean mask over the pool's slots (page * page_size + row) that some
    query of the call may read from the cache: for each sequence with new
    tokens, the cached positions [lo, ctx) where ctx = kv_len - q_len and lo
    is the first key inside the first new token's window (0 without a
    window).  Everything else -- rows past kv_len in the last page, rows
    before the window, the new tokens' own slots before they are written,
    unused pages -- is never read by a correct kernel."""
    mask = np.zeros(w.num_pages * w.page_size, dtype=bool)
    W = w.sliding_window
    for s in range(w.num_seqs):
        q, kv = int(w.q_lens[s]), int(w.kv_lens_valid[s])
        if q == 0:
            continue
        ctx = kv - q
        lo = max(0, ctx - W + 1) if W else 0
        pos = np.arange(lo, ctx, dtype=np.int64)
        pages = w.block_tables[s * w.pages_per_seq + pos // w.page_size].astype(np.int64)
        mask[pages * w.page_size + pos % w.page_size] = True
    return mask


def poison_unread_slots(w, pool: torch.Tensor) -> torch.Tensor:
    """A copy of the CPU pool whose unread slots (see read_slots) hold
    non-finite bit patterns, cycling over NONFINITE_BF16 / NONFINITE_E4M3
    element by element."""
    out = pool.clone()
    rows = w.num_pages * w.page_size
    unread = torch.from_numpy(~read_slots(w))
    if w.kv_dtype == "fp8":
        flat = out.view(torch.uint8).view(rows, -1)
        pat = torch.tensor(NONFINITE_E4M3, dtype=torch.uint8)
    else:
        flat = out.view(torch.int16).view(rows, -1)
        pat = torch.tensor([np.int16(np.uint16(x).view(np.int16)) for x in NONFINITE_BF16],
                           dtype=torch.int16)
    n = flat.shape[1]
    fill = pat.repeat(-(-n // len(pat)))[:n]
    flat[unread] = fill
    return out
