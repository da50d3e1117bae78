"""rpa_forward_noalloc, the entry point for callers that cannot allocate.

Some callers cannot hand the library a device workspace: code running inside
an allocator or memory-pool callback (allocating would re-enter the
allocator), plugins of runtimes that own every device allocation, or
deployments that forbid allocation after start-up.  rpa_forward_noalloc
serves them from a fixed device array inside the library.  These tests call
it through the C ABI and check that, call after call, it returns exactly what
rpa_forward returns on the same inputs -- outputs and page pools bit for bit,
since both run the same kernels and the split combine reads its partial
results in a fixed order, so a stale word left in the shared array by an
earlier call would show as a difference -- that one of those calls also
matches the CPU oracle, and that it refuses problems too large for its
array.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import ragged_paged_attention_kv_gb300 as rpa
from helpers import assert_close, run_oracle
from ragged_paged_attention_kv_gb300 import _lib
import workloads as wl

pytestmark = pytest.mark.gpu


def _entry():
    return _lib.load().rpa_forward_noalloc


def _case(name, seed, q_lens, kv_lens, **kw):
    base = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    base.update(kw)
    return wl.make_custom(name, seed, q_lens, kv_lens, **base)


def _inputs(w, dev):
    q, k, v = w.make_qkv()
    sink = w.make_sink()
    d = lambda x: torch.as_tensor(x).to(dev).contiguous()
    meta = [d(w.kv_lens), d(w.block_tables), d(w.query_start_loc), d(w.distribution)]
    return d(q), d(k), d(v), meta, (d(sink) if sink is not None else None), w.make_pool(dev)


def _with_forward(w, q, k, v, meta, sink, pool):
    out = torch.zeros_like(q)
    fp8 = w.kv_dtype == "fp8"
    rpa.forward(q, k, v, pool, *meta, sink, softmax_scale=w.softmax_scale,
                sliding_window=w.sliding_window, logits_soft_cap=w.logits_soft_cap,
                k_scale=w.k_scale if fp8 else None, v_scale=w.v_scale if fp8 else None, out=out)
    return out


def _with_noalloc(w, q, k, v, meta, sink, pool):
    out = torch.zeros_like(q)
    p = rpa.make_params(**w.params())
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _entry()(ctypes.byref(p), ptr(q), ptr(k), ptr(v), ptr(pool), *[ptr(m) for m in meta],
                  ptr(sink), ptr(out), stream)
    assert rc == 0, f"rpa_forward_noalloc returned {rc}"
    return out


def test_noalloc_matches_rpa_forward_call_after_call():
    dev = torch.device("cuda")
    # A: decode splits (partial results in the scratch) plus prefill tiles;
    # B: a smaller problem that runs on whatever A left in the array;
    # then A again.
    cases = [
        _case("na_a", 501, [1] * 10 + [70, 33], [1500, 40, 900, 2200, 1, 300, 1023, 64, 777, 2048, 300, 33],
              has_sink=True, sliding_window=0),
        _case("na_b", 502, [1, 1, 9], [17, 400, 9], num_q_heads=8, num_kv_heads=2, head_dim=64,
              kv_dtype="fp8", k_scale=0.05, v_scale=0.05, logits_soft_cap=30.0, sliding_window=64),
    ]
    for i, w in enumerate((cases[0], cases[1], cases[0])):
        q, k, v, meta, sink, pool = _inputs(w, dev)
        pool_before = pool.cpu()
        pool_ref = pool.clone()
        ref = _with_forward(w, q, k, v, meta, sink, pool_ref)
        got = _with_noalloc(w, q, k, v, meta, sink, pool)
        torch.cuda.synchronize()
        n = w.num_query_tokens
        assert torch.equal(got[:n], ref[:n]), f"{w.name}: outputs differ from rpa_forward"
        assert torch.equal(pool, pool_ref), "page pools differ"
        if i == 0:
            # the first call also against the oracle (so the equality above is
            # not an agreement of two wrong results)
            hq, hk, hv = w.make_qkv()
            ref_out, ref_cache = run_oracle(w, hq, hk, hv, pool_before, w.make_sink())
            assert_close(got[:n].float().cpu().numpy().astype(np.float64), ref_out, w.name)
            assert np.array_equal(pool.cpu().view(torch.uint8).numpy().reshape(-1), ref_cache)


def test_noalloc_refuses_problems_larger_than_its_array():
    p = rpa.make_params(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                        num_pages=1 << 20, pages_per_seq=4096, max_num_seqs=100000,
                        total_tokens=100000)
    assert rpa.workspace_size(p) > (32 << 20)
    z = ctypes.c_void_p(256)
    rc = _entry()(ctypes.byref(p), z, z, z, z, z, z, z, z, None, z, None)
    assert rc == _lib.RPA_ERR_NOALLOC_TOO_LARGE
    assert b"fixed device array" in _lib.load().rpa_status_string(rc)
