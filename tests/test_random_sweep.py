"""Seeded random batches through the CUDA path, each checked against the oracle.

Every case draws its shape and options at random within the library's
envelope: head_dim 64/96/128/192/256, GQA groups 1-16, page sizes 1-256,
bf16 or e4m3 caches (scalar or per-head scales, with or without quantised
queries), sliding windows, soft caps, sinks, and a mix of decode sequences
and prefill sequences (chunked, with cached context, or fresh) in the three
distribution classes.  Some cases hold many short prefill sequences, so the
CTAs of the prefill kernels take several units each, with ragged tails.
The oracle's work per case is capped so the whole sweep runs in well under
a minute.  The generator is checked on the CPU (every case is well formed
and within the cap); the GPU test compares the whole page pool bit for bit
and every output element within the stated tolerance.
"""
import numpy as np
import pytest

import workloads as wl
from helpers import assert_close, pool_bytes, run_oracle

N_CASES = 64
ORACLE_WORK_CAP = 2.5e8  # (query token, visible key) pairs x Hq x D


def _oracle_work(q_lens, kv_lens, window, hq, d):
    pairs = 0
    for q, kv in zip(q_lens, kv_lens):
        for i in range(q):
            pos = kv - q + i
            pairs += min(pos + 1, window) if window else pos + 1
    return pairs * hq * d


def random_case(i):
    rng = np.random.default_rng(7000 + i)
    for _ in range(1000):
        d = int(rng.choice([64, 96, 128, 192, 256]))
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 4, 8, 16]))
        if hkv * g > 64:
            continue
        page = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256]))
        fp8 = bool(rng.random() < 0.5)
        window = int(rng.integers(1, 300)) if rng.random() < 0.35 else 0
        cap = 30.0 if rng.random() < 0.3 else 0.0
        sink = bool(rng.random() < 0.3)
        many = i % 4 == 3  # many short prefill sequences: several units per CTA
        n_dec = int(rng.integers(0, 40))
        n_pf = int(rng.integers(20, 48)) if many else int(rng.integers(0, 10))
        if n_dec + n_pf == 0:
            continue
        q = [1] * n_dec
        kv = [int(rng.integers(1, 600)) for _ in range(n_dec)]
        for _ in range(n_pf):
            ql = int(rng.integers(1, 40)) if many else int(rng.integers(1, 200))
            ctx = int(rng.integers(0, 400)) if rng.random() < 0.7 else 0
            q.append(ql)
            kv.append(ql + ctx)
        if _oracle_work(q, kv, window, hkv * g, d) > ORACLE_WORK_CAP:
            continue
        n_chunk = int(rng.integers(0, n_pf + 1))
        kw = dict(num_q_heads=hkv * g, num_kv_heads=hkv, head_dim=d, page_size=page,
                  sliding_window=window, logits_soft_cap=cap, has_sink=sink,
                  distribution=[n_dec, n_dec + n_chunk, n_dec + n_pf])
        if fp8:
            kw.update(kv_dtype="fp8", k_scale=float(rng.uniform(0.02, 0.3)),
                      v_scale=float(rng.uniform(0.02, 0.3)))
            if rng.random() < 0.3:
                kw.update(k_scale_heads=list(rng.uniform(0.02, 0.3, hkv)),
                          v_scale_heads=list(rng.uniform(0.02, 0.3, hkv)))
            if rng.random() < 0.35:
                kw.update(q_scale=0.02)
        return wl.make_custom(f"rs{i}", 7000 + i, q, kv, **kw)
    raise RuntimeError("no case within the cap")


def test_random_cases_are_well_formed():
    kinds = set()
    for i in range(N_CASES):
        w = random_case(i)
        d = w.distribution
        assert 0 <= d[0] <= d[1] <= d[2] == w.num_seqs <= w.max_num_seqs
        assert np.all(w.q_lens[:d[0]] == 1)
        assert _oracle_work(w.q_lens, w.kv_lens_valid, w.sliding_window, w.num_q_heads,
                            w.head_dim) <= ORACLE_WORK_CAP
        kinds.add((w.head_dim, w.kv_dtype))
    assert len({k[0] for k in kinds}) >= 4 and {k[1] for k in kinds} == {"bf16", "fp8"}


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(i):
    from test_gpu_parity import run_gpu
    w = random_case(i)
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    sink = w.make_sink()
    ref_out, ref_cache = run_oracle(w, q, k, v, pool, sink)
    out, pool_after, status = run_gpu(w, q, k, v, pool, sink)
    assert status == 0, f"status {status:#x}"
    assert np.array_equal(pool_bytes(pool_after), ref_cache), "page pool differs from the oracle"
    assert_close(out[:w.num_query_tokens], ref_out, w.name)
