"""Bounded device waits: a wait that runs out is reported, not hung on.

Every mbarrier wait in the library's TMA / tcgen05 kernels gives up after a
limit (2 s in the product build), sets RPA_STATUS_TIMEOUT in the workspace's
status word, raises a CTA-wide abort flag, lets the copies and tensor-core
products it issued finish, and leaves through its normal exit -- so a stuck
pipeline never hangs the GPU and the context stays usable.

These tests build a separate copy of the library (the product library is not
touched) with a 20 ms limit in which the producers never signal that a unit's
query tile has landed: a flag that nothing sets, so the first wait on it runs
out in every CTA that gets a unit.  Each call must then

* return promptly (the aborting roles see the flag instead of waiting out
  their own limits one after another),
* report RPA_STATUS_TIMEOUT,
* leave every slot of the page pool outside the step's new-token slots
  unchanged (new-token slots hold either their old bytes or exactly the
  value the page write stores),

and afterwards the product library must still compute a correct call in the
same process (the context is usable).  The decode kernel, the tcgen05
prefill for head_dim 128 and for head_dim 256, and an fp8 cache are covered.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import ragged_paged_attention_kv_gb300 as rpa
import workloads as wl
from helpers import assert_close, pool_bytes, run_oracle
from ragged_paged_attention_kv_gb300 import _lib

pytestmark = pytest.mark.gpu

DEV = "cuda"
WAIT_LIMIT_NS = 20_000_000  # 20 ms


@pytest.fixture(scope="module")
def stall_lib():
    from ragged_paged_attention_kv_gb300 import build
    path = build.build(variant="stall_query",
                       defines=[f"-DRPA_WAIT_LIMIT_NS={WAIT_LIMIT_NS}ull",
                                "-DRPA_TEST_STALL_QUERY=1"])
    lib = ctypes.CDLL(path)
    vp, pp = ctypes.c_void_p, ctypes.POINTER(_lib.RpaParams)
    lib.rpa_workspace_size.argtypes = [pp, ctypes.POINTER(ctypes.c_size_t)]
    lib.rpa_workspace_size.restype = ctypes.c_int
    lib.rpa_forward.argtypes = [pp] + [vp] * 11 + [ctypes.c_size_t, vp]
    lib.rpa_forward.restype = ctypes.c_int
    lib.rpa_get_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.rpa_get_status.restype = ctypes.c_int
    return lib


CASES = [
    ("decode_bf16", lambda: wl.make_custom("to1", 601, [1] * 6, [700, 17, 1290, 333, 65, 9],
                                           num_q_heads=32, num_kv_heads=8, head_dim=128,
                                           page_size=16)),
    ("prefill_tc_bf16", lambda: wl.make_custom("to2", 602, [1, 300, 40], [900, 700, 40],
                                               num_q_heads=32, num_kv_heads=8, head_dim=128,
                                               page_size=16)),
    ("prefill_tc_wide", lambda: wl.make_custom("to3", 603, [1, 200, 40], [900, 700, 40],
                                               num_q_heads=16, num_kv_heads=8, head_dim=256,
                                               page_size=16)),
    ("fp8_options", lambda: wl.make_custom("to4", 604, [1, 1, 64, 20], [900, 129, 700, 20],
                                           num_q_heads=64, num_kv_heads=8, head_dim=64,
                                           page_size=16, kv_dtype="fp8", k_scale=0.05,
                                           v_scale=0.07, logits_soft_cap=30.0, has_sink=True,
                                           sliding_window=300)),
]


def _new_token_slots(w):
    rows = np.zeros(w.num_pages * w.page_size, dtype=bool)
    for s in range(w.num_seqs):
        ctx = int(w.kv_lens_valid[s]) - int(w.q_lens[s])
        pos = np.arange(ctx, int(w.kv_lens_valid[s]))
        rows[w.block_tables[s * w.pages_per_seq + pos // w.page_size].astype(np.int64)
             * w.page_size + pos % w.page_size] = True
    return rows


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_wait_that_runs_out_is_reported_promptly(stall_lib, name, make):
    w = make()
    fp8 = w.kv_dtype == "fp8"
    q, k, v = w.make_qkv()
    sink = w.make_sink()
    pool0 = w.make_pool("cpu")
    d = lambda x: torch.as_tensor(x).to(DEV).contiguous()
    dq, dk, dv = d(q), d(k), d(v)
    meta = [d(w.kv_lens), d(w.block_tables), d(w.query_start_loc), d(w.distribution)]
    dsink = d(sink) if sink is not None else None
    pool = pool0.to(DEV)
    out = torch.zeros_like(dq)
    p = rpa.make_params(**w.params())
    n = ctypes.c_size_t(0)
    assert stall_lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    ws = torch.empty(n.value, dtype=torch.uint8, device=DEV)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = stall_lib.rpa_forward(ctypes.byref(p), ptr(dq), ptr(dk), ptr(dv), ptr(pool),
                               *[ptr(m) for m in meta], ptr(dsink), ptr(out), ptr(ws), n.value,
                               stream)
    assert rc == 0
    status = ctypes.c_int32(0)
    assert stall_lib.rpa_get_status(ptr(ws), stream, ctypes.byref(status)) == 0
    elapsed = time.perf_counter() - t0
    assert status.value & _lib.RPA_STATUS_TIMEOUT, f"status {status.value:#x}"
    # a few limits at most (decode, then prefill), far below one product limit
    assert elapsed < 1.0, f"the call took {elapsed:.3f} s"
    # nothing outside the new-token slots changed; those hold the old bytes
    # or exactly what the page write stores
    rows = w.num_pages * w.page_size
    got = pool_bytes(pool.cpu()).reshape(rows, -1)
    before = pool_bytes(pool0).reshape(rows, -1)
    written = oracle.update_cache(oracle.make_params(**w.params()), k, v, pool_bytes(pool0),
                                  w.kv_lens, w.block_tables, w.query_start_loc,
                                  w.num_seqs).reshape(rows, -1)
    new = _new_token_slots(w)
    assert np.array_equal(got[~new], before[~new])
    same = np.all(got[new] == before[new], axis=1) | np.all(got[new] == written[new], axis=1)
    assert np.all(same)
    # the context is still usable: the product library computes a correct call
    ref_out, ref_cache = run_oracle(w, q, k, v, pool0, sink)
    pool2 = pool0.to(DEV)
    out2 = torch.zeros_like(dq)
    ws2 = rpa.alloc_workspace(p, DEV)
    rpa.forward(dq, dk, dv, pool2, *meta, dsink, softmax_scale=w.softmax_scale,
                sliding_window=w.sliding_window, logits_soft_cap=w.logits_soft_cap,
                k_scale=w.k_scale if fp8 else None, v_scale=w.v_scale if fp8 else None,
                out=out2, workspace=ws2)
    assert rpa.get_status(ws2) == 0
    assert np.array_equal(pool_bytes(pool2.cpu()), ref_cache)
    assert_close(out2[:w.num_query_tokens].float().cpu().numpy().astype(np.float64), ref_out,
                 name)
