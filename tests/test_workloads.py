"""Every benchmark workload is a well-formed call (CPU only).

The metadata must be consistent:

- `distribution` holds cumulative class ends, with every sequence counted;
- `query_start_loc` starts at 0, never decreases and fits in total_tokens;
- kv_len >= q_len, within the block table's capacity;
- decode-class sequences have one new token;
- every page a sequence uses lies in the pool and belongs to it alone;
- the same seed gives the same workload.

The library's host checks must accept the parameters, and the benchmark must
have a description for each workload (its JSON line names the workload by it).
"""
import ctypes
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402

NAMES = sorted(wl.WORKLOADS)


@pytest.fixture(scope="module")
def lib():
    from ragged_paged_attention_kv_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


@pytest.mark.parametrize("name", NAMES)
def test_workload_is_well_formed(name, lib):
    import ragged_paged_attention_kv_gb300 as rpa

    w = wl.get(name)
    S = w.num_seqs
    d = [int(x) for x in w.distribution]
    assert 0 <= d[0] <= d[1] <= d[2] == S <= w.max_num_seqs
    qsl = np.asarray(w.query_start_loc, np.int64)
    assert qsl[0] == 0 and np.all(np.diff(qsl) >= 0)
    assert qsl[S] == w.num_query_tokens <= w.total_tokens
    q = np.asarray(w.q_lens, np.int64)
    kv = np.asarray(w.kv_lens_valid, np.int64)
    assert np.all(kv >= q) and np.all(kv <= w.pages_per_seq * w.page_size)
    assert np.all(q[:d[0]] == 1), "decode-class sequences have one new token"
    bt = np.asarray(w.block_tables).reshape(w.max_num_seqs, w.pages_per_seq)
    used = np.concatenate([bt[s, :-(-int(kv[s]) // w.page_size)] for s in range(S)])
    assert used.min() >= 0 and used.max() < w.num_pages
    assert len(np.unique(used)) == len(used), "a page belongs to one sequence"
    again = wl.get(name)
    assert np.array_equal(again.kv_lens_valid, w.kv_lens_valid)
    assert np.array_equal(again.block_tables, w.block_tables)
    p = rpa.make_params(**{k: v for k, v in w.params().items()
                           if k not in ("kv_fp8", "k_scale_heads", "v_scale_heads")},
                        kv_fp8=w.kv_dtype == "fp8")
    n = ctypes.c_size_t(0)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > 0
    assert name in bench.DESCRIPTIONS
