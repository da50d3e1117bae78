"""The benchmark's algorithmic work counts (the roofline numerators), checked
on hand-counted cases.

Decode bytes: every cached key/value row in the window read once (2*Hkv*D
elements of the cache's type per key), the new token's bf16 key/value read
from the inputs and written into its page, the query read and the output
written.  Prefill flops: 4*D*Hq per unmasked (query token, key) pair.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def _one(q_len, kv_len, *, decode, **kw):
    base = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16)
    base.update(kw)
    d0 = 1 if decode else 0
    return wl.make_custom("w", 1, [q_len], [kv_len], distribution=[d0, 1, 1], **base)


def test_decode_sequence_bytes_and_flops():
    w = _one(1, 10, decode=True)
    work = bench.algorithmic_work(w)
    # 9 cached keys x (K + V) x 2 kv heads x 64 x 2 bytes        = 4608
    # new token: bf16 K, V read from the inputs (512) + written to the page (512)
    # query read (4 heads x 64 x 2 = 512) + output written (512)
    assert work["decode"]["bytes"] == 4608 + 1024 + 1024
    # the new token attends to 10 keys; 4 flops x 64 x 4 q-heads per key
    assert work["decode"]["flops"] == 10 * 4 * 64 * 4
    assert work["decode"]["tokens"] == 1
    assert work["prefill"] == {"bytes": 0, "flops": 0, "tokens": 0}


def test_windowed_prefill_counts_only_the_band():
    # positions 2, 3, 4 (ctx = 2) with a 2-key window: each sees 2 keys
    w = _one(3, 5, decode=False, sliding_window=2)
    work = bench.algorithmic_work(w)
    assert work["prefill"]["flops"] == 6 * 4 * 64 * 4
    # cached rows any new token needs: position 1 only (position 0 is out of
    # every window): 1 x 2 x 2 x 64 x 2 = 512; new tokens 3 x 1024; q + out 3 x 1024
    assert work["prefill"]["bytes"] == 512 + 3 * 1024 + 3 * 1024
    assert work["prefill"]["tokens"] == 3


def test_fp8_cache_rows_are_one_byte():
    w = _one(1, 10, decode=True, kv_dtype="fp8", k_scale=0.05, v_scale=0.05)
    # 9 cached keys at 1 byte: 2304; new token: 512 read + 256 written; q + out 1024
    assert bench.algorithmic_work(w)["decode"]["bytes"] == 2304 + 768 + 1024


def test_decode_workload_bytes_match_the_stated_figure():
    w = wl.get("decode")
    b = bench.algorithmic_work(w)["decode"]["bytes"]
    kv = np.asarray(w.kv_lens_valid, np.int64)
    # 256 decode sequences, Hq32/Hkv8/D128, bf16: cached rows sum(kv - 1) x
    # 2 x 8 x 128 x 2 bytes; per new token 8 KB of K/V (read + page write) and
    # 16 KB of query + output
    assert b == int((kv - 1).sum()) * 4096 + 256 * (8192 + 16384)
    assert b == pytest.approx(2.364e9, rel=1e-3)
