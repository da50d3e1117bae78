"""GPU parity: librpa.so against the CPU oracle (needs a GB300).

Every case calls the C ABI (through the ctypes binding) on seeded inputs and
compares with the oracle on the same inputs:
  * the whole page pool after the call, bit for bit (new slots written, every
    other byte untouched);
  * the attention output, element by element: the error beyond half a bf16
    ulp of the exact value (the rounding any bf16 output carries) is at most
    1e-2, and the mean absolute difference from the fp64 oracle at most 1e-3.
Small cases span several tiles, several decode splits and ragged tails;
the full-size workloads are checked on sampled sequences/tokens in the
launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import ragged_paged_attention_kv_gb300 as rpa
from helpers import assert_close, bf16_half_ulp, poison_unread_slots, pool_bytes, run_oracle
import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV).contiguous()


def run_gpu(w, q, k, v, pool_before, sink=None, workspace=None, out=None):
    """One rpa_forward on copies of the inputs; returns (out cpu, pool cpu, status)."""
    pool = pool_before.to(DEV).clone()
    out_t = out if out is not None else torch.full((w.total_tokens, w.num_q_heads, w.head_dim),
                                                   7.0, dtype=torch.bfloat16, device=DEV)
    params = rpa.make_params(**{k_: v_ for k_, v_ in w.params().items()
                                if k_ not in ("kv_fp8", "k_scale_heads", "v_scale_heads")},
                             kv_fp8=w.kv_dtype == "fp8")
    ws = workspace if workspace is not None else rpa.alloc_workspace(params, DEV)
    fp8 = w.kv_dtype == "fp8"
    # per-kv-head scales go to the library as float32 device tensors
    ks = _dev(w.k_scale_heads, torch.float32) if w.k_scale_heads is not None else \
        (w.k_scale if fp8 else None)
    vs = _dev(w.v_scale_heads, torch.float32) if w.v_scale_heads is not None else \
        (w.v_scale if fp8 else None)
    rpa.forward(_dev(q), _dev(k), _dev(v), pool, _dev(w.kv_lens), _dev(w.block_tables),
                _dev(w.query_start_loc), _dev(w.distribution),
                None if sink is None else _dev(sink),
                softmax_scale=w.softmax_scale, sliding_window=w.sliding_window,
                logits_soft_cap=w.logits_soft_cap, k_scale=ks, v_scale=vs, q_scale=w.q_scale,
                out=out_t, workspace=ws)
    status = rpa.get_status(ws)
    torch.cuda.synchronize()
    return out_t.float().cpu().numpy().astype(np.float64), pool.cpu(), status


def check_case(w, expect_status=0, poison=False):
    """poison: the slots no query may read hold NaN / Inf bit patterns."""
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    if poison:
        pool = poison_unread_slots(w, pool)
    sink = w.make_sink()
    ref_out, ref_cache = run_oracle(w, q, k, v, pool, sink)
    out, pool_after, status = run_gpu(w, q, k, v, pool, sink)
    assert status == expect_status, f"status {status:#x}"
    assert np.array_equal(pool_bytes(pool_after), ref_cache), "page pool differs from the oracle"
    n = w.num_query_tokens
    assert_close(out[:n], ref_out, w.name)
    # rows past query_start_loc[S] stay untouched
    assert np.all(out[n:] == 7.0)
    return out[:n], ref_out


def _case(name, seed, q_lens, kv_lens, **kw):
    base = dict(num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16)
    base.update(kw)
    return wl.make_custom(name, seed, q_lens, kv_lens, **base)


def test_tiny_workload():
    check_case(wl.tiny())


CASES = [
    # decode only, several splits per sequence (combine path), long and short
    ("decode_splits", lambda: _case("ds", 101, [1] * 6, [700, 17, 1, 16, 33, 1290],
                                    num_q_heads=32, num_kv_heads=8, head_dim=128)),
    ("decode_g1_d64", lambda: _case("d1", 102, [1] * 5, [5, 64, 65, 300, 513],
                                    num_q_heads=4, num_kv_heads=4)),
    ("decode_g16", lambda: _case("d16", 103, [1] * 3, [100, 260, 31], num_q_heads=32,
                                 num_kv_heads=2, head_dim=128, page_size=32)),
    # prefill with many tiles and ragged tails, fresh and with context
    ("prefill_fresh", lambda: _case("pf", 104, [150, 37], [150, 37], num_q_heads=16,
                                    num_kv_heads=4, head_dim=128)),
    ("prefill_chunk", lambda: _case("pc", 105, [70, 5, 129], [300, 260, 129], page_size=64)),
    ("mixed_classes", lambda: _case("mx", 106, [1, 1, 1, 40, 9, 77], [90, 300, 2, 140, 9, 200],
                                    num_q_heads=32, num_kv_heads=4, head_dim=128,
                                    distribution=[3, 5, 6])),
    ("q_len_zero", lambda: _case("qz", 107, [0, 3, 0, 1], [12, 30, 1, 7], distribution=[0, 0, 4])),
    ("page_size_1", lambda: _case("p1", 108, [1, 6], [40, 20], page_size=1)),
    ("page_size_256", lambda: _case("p256", 109, [1, 20], [600, 530], page_size=256)),
    # options
    ("window", lambda: _case("w", 110, [1, 1, 50, 100], [600, 20, 70, 300], sliding_window=37)),
    ("window_pagealigned", lambda: _case("wp", 111, [1, 64], [512, 256], sliding_window=64,
                                         head_dim=128)),
    ("softcap", lambda: _case("sc", 112, [1, 33], [400, 120], logits_soft_cap=5.0,
                              softmax_scale=0.6)),
    ("sink", lambda: _case("sk", 113, [1, 1, 45], [333, 2, 45], has_sink=True)),
    ("fp8", lambda: _case("f8", 114, [1, 1, 30, 8], [500, 3, 100, 8], kv_dtype="fp8",
                          k_scale=0.05, v_scale=0.05)),
    ("fp8_all_options", lambda: _case("f8a", 115, [1, 1, 1, 64, 20], [900, 129, 5, 200, 20],
                                      kv_dtype="fp8", k_scale=0.05, v_scale=0.07, num_q_heads=64,
                                      num_kv_heads=8, head_dim=64, logits_soft_cap=30.0,
                                      has_sink=True, sliding_window=128, softmax_scale=0.125)),
    ("fp8_d128", lambda: _case("f8d", 116, [1, 17], [260, 80], kv_dtype="fp8", k_scale=0.3,
                               v_scale=0.1, head_dim=128)),
    ("padding_rows", lambda: _case("pad", 117, [1, 5], [9, 12], max_num_seqs=5, extra_tokens=6,
                                   pages_per_seq=4)),
    # per-kv-head fp8 scales: decode splits, the tcgen05 prefill (head_dim 64
    # and 128), the mma.sync prefill (pages of 4 rows), with every option
    ("fp8_per_head", lambda: _case("fh", 118, [1, 1, 40, 9], [1400, 70, 300, 9],
                                   kv_dtype="fp8", num_q_heads=16, num_kv_heads=4,
                                   k_scale_heads=[0.02, 0.05, 0.11, 0.3],
                                   v_scale_heads=[0.07, 0.015, 0.2, 0.05])),
    ("fp8_per_head_d128_options", lambda: _case(
        "fhd", 119, [1, 1, 130, 33], [800, 40, 400, 33], kv_dtype="fp8", num_q_heads=16,
        num_kv_heads=2, head_dim=128, k_scale_heads=[0.04, 0.09], v_scale_heads=[0.12, 0.03],
        logits_soft_cap=20.0, has_sink=True, sliding_window=200)),
    ("fp8_per_head_p4", lambda: _case("fh4", 120, [1, 25], [90, 60], kv_dtype="fp8",
                                      page_size=4, k_scale_heads=[0.06, 0.02],
                                      v_scale_heads=[0.03, 0.08])),
    ("fp8_per_head_k_only", lambda: _case("fhk", 121, [1, 12], [300, 50], kv_dtype="fp8",
                                          k_scale=0.05, v_scale=0.05,
                                          k_scale_heads=[0.03, 0.07])),
    # head_dim 256: decode (query fragments re-read from a padded slot) and
    # the warp-level MMA prefill
    ("d256_decode_splits", lambda: _case("e1", 122, [1] * 6, [700, 17, 1, 16, 33, 1290],
                                         num_q_heads=16, num_kv_heads=8, head_dim=256)),
    ("d256_prefill", lambda: _case("e2", 123, [150, 37, 1, 64], [150, 300, 90, 64],
                                   num_q_heads=8, num_kv_heads=4, head_dim=256)),
    ("d256_gemma_options", lambda: _case("e3", 124, [1, 1, 40, 9], [300, 5, 140, 9],
                                         num_q_heads=16, num_kv_heads=8, head_dim=256,
                                         sliding_window=64, logits_soft_cap=50.0,
                                         has_sink=True, softmax_scale=0.0625,
                                         distribution=[2, 3, 4])),
    ("d256_fp8", lambda: _case("e4", 125, [1, 1, 30, 8], [500, 3, 100, 8], kv_dtype="fp8",
                               k_scale=0.05, v_scale=0.07, head_dim=256, num_q_heads=8,
                               num_kv_heads=2)),
    ("d256_fp8_per_head_p64", lambda: _case("e5", 126, [1, 1, 70], [900, 64, 200],
                                            kv_dtype="fp8", head_dim=256, page_size=64,
                                            k_scale_heads=[0.04, 0.1], v_scale_heads=[0.06, 0.02],
                                            has_sink=True)),
    ("d256_g16_p4", lambda: _case("e6", 127, [1, 1, 20], [260, 7, 45], num_q_heads=32,
                                  num_kv_heads=2, head_dim=256, page_size=4)),
    # head_dim 96 (run as 128 with zero columns) and 192 (three 64-column blocks)
    ("d96_decode_prefill", lambda: _case("e7", 128, [1, 1, 1, 40, 9], [700, 17, 300, 140, 9],
                                         num_q_heads=32, num_kv_heads=8, head_dim=96,
                                         distribution=[3, 4, 5])),
    ("d96_mha_options", lambda: _case("e8", 129, [1, 1, 33], [1290, 2, 120], num_q_heads=4,
                                      num_kv_heads=4, head_dim=96, sliding_window=100,
                                      logits_soft_cap=30.0, has_sink=True)),
    ("d96_fp8", lambda: _case("e9", 130, [1, 1, 30, 8], [500, 3, 100, 8], kv_dtype="fp8",
                              k_scale=0.05, v_scale=0.07, head_dim=96)),
    ("d96_p1", lambda: _case("e10", 131, [1, 6], [40, 20], head_dim=96, page_size=1)),
    ("d192_decode_prefill", lambda: _case("e11", 132, [1, 1, 70, 5], [900, 64, 200, 260],
                                          num_q_heads=16, num_kv_heads=4, head_dim=192)),
    ("d192_fp8_options", lambda: _case("e12", 133, [1, 1, 20], [600, 33, 45], kv_dtype="fp8",
                                       head_dim=192, k_scale_heads=[0.04, 0.1],
                                       v_scale_heads=[0.06, 0.02], logits_soft_cap=20.0,
                                       sliding_window=150, page_size=32)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_small_cases(name, make):
    check_case(make())


def _tc(name, seed, q_lens, kv_lens, **kw):
    """A case that takes the tcgen05 prefill path (bf16 cache, head_dim 128, P >= 8)."""
    base = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    base.update(kw)
    return wl.make_custom(name, seed, q_lens, kv_lens, **base)


TC_CASES = [
    ("p8", lambda: _tc("t8", 201, [1, 90, 13], [70, 400, 141], page_size=8)),
    ("p128", lambda: _tc("t128", 202, [1, 200, 7], [900, 700, 135], page_size=128)),
    ("p256_partial_pages", lambda: _tc("t256", 203, [150, 40], [1000, 40], page_size=256)),
    ("p1024", lambda: _tc("t1k", 204, [1, 130], [1500, 1200], page_size=1024)),
    ("gqa1_long_tiles", lambda: _tc("tg1", 205, [300, 129, 1], [900, 129, 50], num_q_heads=4,
                                    num_kv_heads=4)),
    ("gqa16", lambda: _tc("tg16", 206, [1, 37, 9], [260, 300, 9], num_q_heads=32,
                          num_kv_heads=2)),
    ("window_in_cached_tiles", lambda: _tc("tw", 207, [1, 100, 64], [2000, 1500, 64],
                                           sliding_window=200)),
    ("window_short", lambda: _tc("tws", 208, [70, 1], [600, 333], sliding_window=5)),
    # windows above 256 keys stay on the tcgen05 kernel (shorter ones run on
    # the warp-level kernel): a window start inside a cached tile
    ("window_300_cached", lambda: _tc("tw3", 212, [1, 100, 64, 300], [2000, 1500, 64, 900],
                                      sliding_window=300)),
    ("softcap_sink", lambda: _tc("tcs", 209, [1, 90, 33], [500, 300, 33], logits_soft_cap=7.5,
                                 has_sink=True, softmax_scale=0.2)),
    ("ctx_tile_aligned", lambda: _tc("tca", 210, [128, 1], [384, 129], page_size=32)),
    ("many_tiles_ragged", lambda: _tc("tmr", 211, [517, 3, 1], [1800, 700, 60], page_size=64)),
]


@pytest.mark.parametrize("name,make", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tcgen05_prefill_cases(name, make):
    check_case(make())


# Slots that no query may read -- rows past kv_len in a sequence's last page,
# rows before the window, the new tokens' slots before they are written,
# unused pages -- hold NaN / Inf bit patterns (bf16 0x7FC0, 0x7F80, 0xFF80,
# 0xFFC1; e4m3 0x7F, 0xFF).  A serving pool holds arbitrary bytes there (the
# ejkernel ragged_page_attention_v3 docstring: only the first num_seqs
# entries of kv_lens / block_tables are valid).  The outputs must stay finite
# and within tolerance and the pool bit-exact, on every kernel path: the
# decode kernel, the tcgen05 prefill (bf16 and fp8 staging) and the
# warp-level MMA prefill (pages of 4 rows; head_dim 256).
POISON_CASES = [
    ("decode_window_splits", lambda: _case("z1", 301, [1] * 6, [700, 17, 1290, 333, 65, 1],
                                           num_q_heads=32, num_kv_heads=8, head_dim=128,
                                           sliding_window=100)),
    ("decode_partial_pages", lambda: _case("z2", 302, [1] * 5, [700, 17, 1290, 333, 65],
                                           num_q_heads=32, num_kv_heads=8, head_dim=128)),
    ("decode_fp8_window_options", lambda: _case("z3", 303, [1] * 5, [900, 129, 5, 2000, 77],
                                                kv_dtype="fp8", k_scale=0.05, v_scale=0.07,
                                                num_q_heads=64, num_kv_heads=8,
                                                logits_soft_cap=30.0, has_sink=True,
                                                sliding_window=128)),
    ("decode_d256_window", lambda: _case("z4", 304, [1] * 4, [300, 5, 1300, 90], num_q_heads=16,
                                         num_kv_heads=8, head_dim=256, sliding_window=64)),
    ("tc_prefill_window_cached", lambda: _tc("z5", 305, [1, 100, 64, 200], [2000, 1500, 64, 700],
                                             sliding_window=200)),
    ("tc_prefill_partial_pages", lambda: _tc("z6", 306, [130, 1, 7], [1000, 70, 135],
                                             page_size=64)),
    ("tc_prefill_p256_window", lambda: _tc("z7", 307, [150, 40], [1000, 40], page_size=256,
                                           sliding_window=300)),
    ("tc_prefill_fp8_options", lambda: _case("z8", 308, [1, 1, 64, 20], [900, 129, 200, 20],
                                             kv_dtype="fp8", k_scale=0.05, v_scale=0.07,
                                             num_q_heads=64, num_kv_heads=8,
                                             logits_soft_cap=30.0, has_sink=True,
                                             sliding_window=128)),
    ("tc_prefill_fp8_d128_window", lambda: _case("z9", 309, [1, 90, 33], [600, 500, 33],
                                                 kv_dtype="fp8", k_scale=0.3, v_scale=0.1,
                                                 head_dim=128, sliding_window=77)),
    ("mma_prefill_p4_window", lambda: _case("z10", 310, [1, 25, 9], [90, 60, 40], page_size=4,
                                            sliding_window=20)),
    # windows above 256 keys: the tcgen05 kernels (bf16 and fp8 staging)
    ("tc_prefill_window_300", lambda: _tc("z14", 314, [1, 100, 64, 300], [2000, 1500, 64, 900],
                                          sliding_window=300)),
    ("tc_prefill_fp8_window_300", lambda: _case("z15", 315, [1, 1, 64, 20], [900, 129, 800, 20],
                                                kv_dtype="fp8", k_scale=0.05, v_scale=0.07,
                                                num_q_heads=64, num_kv_heads=8,
                                                logits_soft_cap=30.0, has_sink=True,
                                                sliding_window=300)),
    ("tcw_prefill_d256_fp8_window_260", lambda: _case("z16", 316, [1, 70, 8], [900, 600, 8],
                                                      kv_dtype="fp8", head_dim=256, k_scale=0.05,
                                                      v_scale=0.07, sliding_window=260)),
    ("mma_prefill_d256_p4_window", lambda: _case("z11", 311, [1, 70, 8], [900, 200, 8],
                                                 head_dim=256, page_size=4, sliding_window=50)),
    ("tcw_prefill_d256_fp8_window", lambda: _case("z12", 312, [1, 70, 8], [900, 200, 8],
                                                  kv_dtype="fp8", head_dim=256, k_scale=0.05,
                                                  v_scale=0.07, sliding_window=50)),
    ("tcw_prefill_d192_partial_pages", lambda: _case("z13", 313, [130, 1, 7], [1000, 70, 135],
                                                     head_dim=192, num_q_heads=16,
                                                     num_kv_heads=8, page_size=64,
                                                     sliding_window=300)),
    # quantised queries: cached key codes go to the tensor core as they are
    ("tc_q8_d128_window_partial_pages", lambda: _case("z17", 317, [1, 90, 33], [600, 500, 35],
                                                      kv_dtype="fp8", k_scale=0.3, v_scale=0.1,
                                                      q_scale=0.02, head_dim=128,
                                                      page_size=64, sliding_window=300)),
    ("tcw_q8_d256_p8_window", lambda: _case("z19", 319, [1, 90, 33], [600, 500, 35],
                                            kv_dtype="fp8", k_scale=0.3, v_scale=0.1,
                                            q_scale=0.02, head_dim=256, num_q_heads=16,
                                            num_kv_heads=8, page_size=8, sliding_window=150)),
    ("tc_q8_d64_options", lambda: _case("z18", 318, [1, 1, 64, 20], [900, 129, 200, 21],
                                        kv_dtype="fp8", k_scale=0.05, v_scale=0.07,
                                        q_scale=0.02, num_q_heads=64, num_kv_heads=8,
                                        logits_soft_cap=30.0, has_sink=True, page_size=8)),
]


@pytest.mark.parametrize("name,make", POISON_CASES, ids=[c[0] for c in POISON_CASES])
def test_nonfinite_bytes_in_unread_slots(name, make):
    check_case(make(), poison=True)


def _tcw(name, seed, q_lens, kv_lens, **kw):
    """A case for the tcgen05 prefill at head_dim 192/256 (one query tile per
    unit, 64-key tiles, S double-buffered in tensor memory)."""
    base = dict(num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16)
    base.update(kw)
    return wl.make_custom(name, seed, q_lens, kv_lens, **base)


TCW_CASES = [
    ("p8", lambda: _tcw("w8", 401, [1, 90, 13], [70, 400, 141], page_size=8)),
    ("p128", lambda: _tcw("w128", 402, [1, 200, 7], [900, 700, 135], page_size=128)),
    ("d192_p256_partial_pages", lambda: _tcw("w256p", 403, [150, 40], [1000, 40], head_dim=192,
                                             page_size=256)),
    ("gqa1_long_tiles", lambda: _tcw("wg1", 404, [300, 129, 1], [900, 129, 50], num_q_heads=4,
                                     num_kv_heads=4)),
    ("gqa16", lambda: _tcw("wg16", 405, [1, 37, 9], [260, 300, 9], num_q_heads=32,
                           num_kv_heads=2)),
    ("window_in_cached_tiles", lambda: _tcw("ww", 406, [1, 100, 64], [2000, 1500, 64],
                                            sliding_window=200)),
    ("window_short", lambda: _tcw("wws", 407, [70, 1], [600, 333], sliding_window=5)),
    ("window_300_cached", lambda: _tcw("ww3", 414, [1, 100, 64, 200], [2000, 1500, 64, 900],
                                       sliding_window=300)),
    ("fp8_window_270", lambda: _tcw("wf82", 415, [1, 90, 20], [900, 700, 20], kv_dtype="fp8",
                                    k_scale=0.05, v_scale=0.07, logits_soft_cap=30.0,
                                    has_sink=True, sliding_window=270)),
    ("softcap_sink", lambda: _tcw("wcs", 408, [1, 90, 33], [500, 300, 33], logits_soft_cap=7.5,
                                  has_sink=True, softmax_scale=0.2)),
    ("ctx_tile_aligned", lambda: _tcw("wca", 409, [128, 1], [384, 129], page_size=32)),
    ("many_tiles_ragged", lambda: _tcw("wmr", 410, [517, 3, 1], [1800, 700, 60], page_size=64,
                                       head_dim=192)),
    ("fp8_options", lambda: _tcw("wf8", 411, [1, 1, 64, 20], [900, 129, 200, 20], kv_dtype="fp8",
                                 k_scale=0.05, v_scale=0.07, logits_soft_cap=30.0, has_sink=True,
                                 sliding_window=128)),
    ("fp8_d192_per_head", lambda: _tcw("wf8h", 412, [1, 90, 33], [600, 500, 33], head_dim=192,
                                       kv_dtype="fp8", k_scale_heads=[0.02, 0.05, 0.11, 0.3,
                                                                      0.04, 0.07, 0.2, 0.09],
                                       v_scale_heads=[0.07, 0.015, 0.2, 0.05, 0.1, 0.03, 0.06,
                                                      0.12])),
    ("fp8_new_tokens_only", lambda: _tcw("wf8n", 413, [200, 70], [200, 70], kv_dtype="fp8",
                                         k_scale=0.3, v_scale=0.1, num_q_heads=8,
                                         num_kv_heads=2)),
]


@pytest.mark.parametrize("name,make", TCW_CASES, ids=[c[0] for c in TCW_CASES])
def test_tcgen05_wide_prefill_cases(name, make):
    check_case(make())


# Quantised queries (q_scale, w8a8): every kernel path with an e4m3 cache --
# decode at head_dim 64 / 96 (one bulk copy per query row) / 128 / 256
# (query fragments re-read from shared memory), the tcgen05 prefill at 64
# and 128, the head_dim 192/256 tcgen05 prefill, and the warp-level MMA
# prefill (pages of 4 rows) -- with per-head scales and every option.
def _q8(name, seed, q_lens, kv_lens, **kw):
    base = dict(num_q_heads=16, num_kv_heads=4, head_dim=64, page_size=16, kv_dtype="fp8",
                k_scale=0.05, v_scale=0.07, q_scale=0.02)
    base.update(kw)
    return wl.make_custom(name, seed, q_lens, kv_lens, **base)


Q8_CASES = [
    ("decode_d64_options", lambda: _q8("q1", 501, [1] * 5, [900, 129, 5, 2000, 77],
                                       num_q_heads=64, num_kv_heads=8, logits_soft_cap=30.0,
                                       has_sink=True, sliding_window=128)),
    ("decode_d128_per_head_splits", lambda: _q8("q2", 502, [1] * 4, [1400, 70, 3000, 9],
                                                head_dim=128, k_scale_heads=[0.02, 0.05, 0.11, 0.3],
                                                v_scale_heads=[0.07, 0.015, 0.2, 0.05])),
    ("decode_d96", lambda: _q8("q3", 503, [1] * 3, [500, 3, 100], head_dim=96)),
    ("decode_d256", lambda: _q8("q4", 504, [1] * 3, [700, 17, 1290], head_dim=256,
                                num_q_heads=16, num_kv_heads=8)),
    ("tc_prefill_d64_mixed", lambda: _q8("q5", 505, [1, 1, 64, 20], [900, 129, 200, 20],
                                         num_q_heads=64, num_kv_heads=8, logits_soft_cap=30.0,
                                         has_sink=True)),
    ("tc_prefill_d128_tiles", lambda: _q8("q6", 506, [1, 300, 33], [800, 700, 33],
                                          head_dim=128, num_q_heads=32, num_kv_heads=8,
                                          sliding_window=300)),
    ("tcw_prefill_d256_per_head", lambda: _q8("q7", 507, [1, 90, 33], [600, 500, 33],
                                              head_dim=256, num_q_heads=16, num_kv_heads=2,
                                              k_scale_heads=[0.04, 0.1],
                                              v_scale_heads=[0.06, 0.02], has_sink=True)),
    ("tcw_prefill_d192", lambda: _q8("q8", 508, [1, 70, 8], [900, 200, 8], head_dim=192,
                                     num_q_heads=8, num_kv_heads=2, logits_soft_cap=20.0)),
    ("mma_prefill_p4", lambda: _q8("q9", 509, [1, 25, 9], [90, 60, 40], page_size=4,
                                   sliding_window=20)),
    # Q K^T on the e4m3 codes (tcgen05 prefill, head_dim 64 / 128): pages
    # larger than a key tile, per-head scales, 8-token pages (the smallest
    # page box of the code tiles), a window and a soft cap, and a long
    # cached context with several new key tiles
    ("tc_q8_d128_per_head_p256", lambda: _q8("q10", 510, [1, 260, 7], [1300, 900, 300],
                                             head_dim=128, num_q_heads=32, num_kv_heads=4,
                                             page_size=256,
                                             k_scale_heads=[0.03, 0.06, 0.1, 0.2],
                                             v_scale_heads=[0.05, 0.02, 0.08, 0.04])),
    ("tc_q8_d64_p8_per_head_window", lambda: _q8("q11", 511, [3, 140, 1], [700, 400, 50],
                                                 head_dim=64, num_q_heads=16, num_kv_heads=2,
                                                 page_size=8, k_scale_heads=[0.03, 0.09],
                                                 v_scale_heads=[0.05, 0.02], sliding_window=200,
                                                 logits_soft_cap=25.0)),
    ("tc_q8_d128_long_cached", lambda: _q8("q12", 512, [600, 1], [2000, 333], head_dim=128,
                                           num_q_heads=8, num_kv_heads=2, page_size=32,
                                           has_sink=True)),
    ("tc_q8_d64_p128_many_units", lambda: _q8("q13", 513, [130, 70, 1, 257],
                                              [1000, 70, 600, 900], head_dim=64,
                                              num_q_heads=32, num_kv_heads=8, page_size=128,
                                              sliding_window=500)),
    # the same on the head_dim 192/256 prefill (64-byte code blocks)
    ("tcw_q8_d192_many_units", lambda: _q8("q14", 514, [70] * 10 + [3] * 30,
                                           [300 + 41 * i for i in range(10)] +
                                           [40 + 23 * i for i in range(30)],
                                           head_dim=192, num_q_heads=16, num_kv_heads=4,
                                           page_size=16, logits_soft_cap=25.0)),
]


@pytest.mark.parametrize("name,make", Q8_CASES, ids=[c[0] for c in Q8_CASES])
def test_quantised_query_cases(name, make):
    check_case(make())


# More units than CTAs, with ragged tails: the planner emits each (sequence,
# head)'s tail unit (often a single query tile) ahead of its full units, so
# CTAs take tail units and full units one after another, and the tails'
# tile counts are odd and even.
MANY_UNIT_CASES = [
    ("bf16_d128", lambda: _case("mu1", 901, [130] * 12 + [2] * 30,
                                [230, 430, 830, 260, 388, 1000, 131, 700, 515, 977, 300, 250]
                                + [100 + 37 * i for i in range(30)],
                                num_q_heads=32, num_kv_heads=8, head_dim=128)),
    ("fp8_d64", lambda: _case("mu2", 902, [40] * 20 + [3] * 24,
                              [100 + 61 * i for i in range(20)] + [50 + 90 * i for i in range(24)],
                              num_q_heads=64, num_kv_heads=8, head_dim=64, kv_dtype="fp8",
                              k_scale=0.05, v_scale=0.07, has_sink=True)),
    ("fp8_q8_d128", lambda: _case("mu3", 903, [130] * 12 + [2] * 30,
                                  [230, 430, 830, 260, 388, 1000, 131, 700, 515, 977, 300, 250]
                                  + [100 + 37 * i for i in range(30)],
                                  num_q_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="fp8",
                                  k_scale=0.05, v_scale=0.07, q_scale=0.02)),
]


@pytest.mark.parametrize("name,make", MANY_UNIT_CASES, ids=[c[0] for c in MANY_UNIT_CASES])
def test_many_units_with_ragged_tails(name, make):
    check_case(make())


# The planner lets the decode kernel leave part of the SMs to the prefill
# kernel when the prefill's flops reach 32 per byte of keys/values the decode
# reads (header word 6 of the workspace).  Both sides of that decision, with
# parity: a few decode sequences beside a large prefill (shared), and many
# decode sequences beside a short chunk (not shared).
SHARE_CASES = [
    ("shared_bf16", True, lambda: _case("sh1", 911, [1] * 6 + [700, 300],
                                        [300, 41, 1000, 77, 129, 640, 900, 300],
                                        num_q_heads=32, num_kv_heads=8, head_dim=128,
                                        distribution=[6, 6, 8])),
    ("shared_fp8_window", True, lambda: _case("sh2", 912, [1] * 40 + [256] * 3,
                                              [200 + 37 * i for i in range(40)] + [900, 400, 256],
                                              num_q_heads=64, num_kv_heads=8, head_dim=64,
                                              kv_dtype="fp8", k_scale=0.05, v_scale=0.05,
                                              sliding_window=128, logits_soft_cap=30.0,
                                              has_sink=True, distribution=[40, 43, 43])),
    ("not_shared", False, lambda: _case("sh3", 913, [1] * 64 + [4],
                                        [2000 + 13 * i for i in range(64)] + [100],
                                        num_q_heads=32, num_kv_heads=8, head_dim=128,
                                        distribution=[64, 65, 65])),
]


@pytest.mark.parametrize("name,shared,make", SHARE_CASES, ids=[c[0] for c in SHARE_CASES])
def test_decode_and_prefill_share_the_sms(name, shared, make):
    w = make()
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    sink = w.make_sink()
    ref_out, ref_cache = run_oracle(w, q, k, v, pool, sink)
    params = rpa.make_params(**{k_: v_ for k_, v_ in w.params().items()
                                if k_ not in ("kv_fp8", "k_scale_heads", "v_scale_heads")},
                             kv_fp8=w.kv_dtype == "fp8")
    ws = rpa.alloc_workspace(params, DEV)
    out, pool_after, status = run_gpu(w, q, k, v, pool, sink, workspace=ws)
    assert status == 0, f"status {status:#x}"
    assert int(ws[:32].view(torch.int32)[6].item()) == int(shared)
    assert np.array_equal(pool_bytes(pool_after), ref_cache)
    assert_close(out[:w.num_query_tokens], ref_out, name)


def test_decode_split_boundaries():
    # kv lengths at page and split boundaries, all decode, big enough batch that
    # the planner's split size stays at its minimum
    kv = [255, 256, 257, 511, 512, 513, 16, 15, 17, 1024, 1025, 2048]
    check_case(_case("db", 121, [1] * len(kv), kv, num_q_heads=16, num_kv_heads=4, head_dim=128))


def test_distribution_only_selects_tiles():
    # decode-class sequences go through the decode kernel, the others through
    # the prefill kernel: the two tile shapes sum in different orders, so the
    # results agree up to rounding, and each matches the oracle
    w = _case("dist", 122, [1, 1, 12, 1], [40, 9, 30, 77])
    outs = []
    for dist in ([2, 2, 4], [0, 0, 4], [0, 2, 4]):
        w.distribution = np.array(dist, np.int32)
        out, ref = check_case(w)
        outs.append(out)
    for o in outs[1:]:
        assert np.max(np.maximum(np.abs(o - outs[0]) - 2 * bf16_half_ulp(ref), 0)) <= 2e-2
        assert np.mean(np.abs(o - outs[0])) <= 2e-3


def test_repeated_calls_match_oracle_every_time():
    """Short units with cached and new key tiles, run repeatedly on fresh
    workspaces: a pipeline race shows up as an occasional wrong call."""
    w = _case("rr", 125, [1] * 10 + [70, 33],
              [1500, 40, 900, 2200, 1, 300, 1023, 64, 777, 2048, 300, 33],
              num_q_heads=32, num_kv_heads=8, head_dim=128, has_sink=True)
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    sink = w.make_sink()
    ref, ref_cache = run_oracle(w, q, k, v, pool, sink)
    n = w.num_query_tokens
    for it in range(10):
        out, pool_after, status = run_gpu(w, q, k, v, pool, sink)
        assert status == 0
        assert np.array_equal(pool_bytes(pool_after), ref_cache)
        assert_close(out[:n], ref, f"call {it}")


def test_decode_class_with_long_query_is_flagged_and_computed():
    w = _case("dq", 123, [1, 3, 1], [30, 10, 5], distribution=[3, 3, 3])
    check_case(w, expect_status=oracle_status_decode_qlen())


def oracle_status_decode_qlen():
    from ragged_paged_attention_kv_gb300 import _lib
    return _lib.RPA_STATUS_DECODE_QLEN


def test_repeat_calls_reuse_workspace():
    w = _case("rep", 124, [1, 1, 20], [300, 1000, 50], num_q_heads=16, num_kv_heads=4)
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    params = rpa.make_params(**{a: b for a, b in w.params().items() if a != "kv_fp8"})
    ws = rpa.alloc_workspace(params, DEV)
    o1, p1, s1 = run_gpu(w, q, k, v, pool, workspace=ws)
    o2, p2, s2 = run_gpu(w, q, k, v, pool, workspace=ws)
    assert s1 == s2 == 0
    assert np.array_equal(o1, o2) and torch.equal(p1, p2)


# --------------------------------------------------------------- bad inputs
def _status_of(w, mutate):
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    mutate(w)
    out, pool_after, status = run_gpu(w, q, k, v, pool)
    return status, out, pool, pool_after


# the e4m3 cases also run the page write ahead of the prefill, which reads the
# metadata alongside the planner and must skip what the planner rejects
_KV = {"bf16": {}, "fp8": dict(kv_dtype="fp8", k_scale=0.05, v_scale=0.05)}

@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_bad_page_sets_status_without_fault(kv):
    from ragged_paged_attention_kv_gb300 import _lib
    w = _case("bp", 131, [1, 4], [40, 30], **_KV[kv])

    def mutate(w):
        w.block_tables = w.block_tables.copy()
        w.block_tables[0] = w.num_pages + 5    # decode seq, cached page
        w.block_tables[w.pages_per_seq + 1] = -3  # prefill seq, page of its new tokens
    status, _, _, _ = _status_of(w, mutate)
    assert status & _lib.RPA_STATUS_BAD_PAGE


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_bad_kv_len_and_qsl_skip_sequence(kv):
    from ragged_paged_attention_kv_gb300 import _lib
    w = _case("bk", 132, [1, 4, 3], [40, 30, 9], **_KV[kv])

    def mutate(w):
        w.kv_lens_valid = w.kv_lens_valid.copy()
        w.kv_lens_valid[1] = 2  # < q_len
    status, out, pool, pool_after = _status_of(w, mutate)
    assert status == _lib.RPA_STATUS_BAD_KV_LEN
    qsl = w.query_start_loc
    assert np.all(out[qsl[1]:qsl[2]] == 7.0)  # the skipped sequence's rows untouched
    # ... and its pages: only the other sequences' new-token slots change
    rows = w.num_pages * w.page_size
    got = pool_bytes(pool_after).reshape(rows, -1)
    before = pool_bytes(pool).reshape(rows, -1)
    pages = w.block_tables[w.pages_per_seq:w.pages_per_seq + 2]  # its 30 keys' two pages
    slots = (pages[:, None].astype(np.int64) * w.page_size + np.arange(w.page_size)).ravel()
    slots = slots[(slots >= 0) & (slots < rows)]
    assert np.array_equal(got[slots], before[slots])


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_bad_distribution_plans_nothing(kv):
    from ragged_paged_attention_kv_gb300 import _lib
    w = _case("bd", 133, [1, 4], [40, 30], **_KV[kv])

    def mutate(w):
        w.distribution = np.array([2, 1, 2], np.int32)
    status, out, pool, pool_after = _status_of(w, mutate)
    assert status == _lib.RPA_STATUS_BAD_DISTRIBUTION
    assert np.all(out == 7.0) and torch.equal(pool, pool_after)


def test_bad_per_head_scale_sets_status():
    from ragged_paged_attention_kv_gb300 import _lib
    w = _case("bs", 135, [1, 4], [40, 30], kv_dtype="fp8", k_scale_heads=[0.05, 0.05],
              v_scale_heads=[0.05, 0.05])

    def mutate(w):
        w.v_scale_heads = np.array([0.05, -0.5], np.float32)
    status, _, _, _ = _status_of(w, mutate)
    assert status == _lib.RPA_STATUS_BAD_SCALE


@pytest.mark.parametrize("head_dim", [64, 96, 128, 192, 256])
def test_decode_units_fill_the_workspace_bound(head_dim):
    """65 decode sequences x 8 kv heads, window 1000 starting 63 keys into a
    64-key stage: with the split target of 512 the chunk is 1024 keys and
    every (sequence, head) spans 1063 keys, so each takes two splits -- 1040
    units, more than target + sequences * heads.  The workspace must hold them
    and the results must match the oracle.  Half the units are one-stage tails,
    so the producer often waits on a query slot while the consumers still read
    it: three runs must give bit-identical outputs (the split combine reads the
    partials in a fixed order, so any difference is a race)."""
    S = 65
    kv = [1063 + 64 * (s % 4) for s in range(S)]
    w = _case("wb", 137, [1] * S, kv, num_q_heads=8, num_kv_heads=8, sliding_window=1000,
              head_dim=head_dim)
    first, _ = check_case(w)
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    for _ in range(2):
        again, _, status = run_gpu(w, q, k, v, pool)
        assert status == 0
        assert np.array_equal(again[:S], first), "decode output differs between runs"


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_empty_batch_is_a_no_op(kv):
    """distribution = [0, 0, 0]: no sequence, nothing planned, nothing written
    (with an e4m3 cache the page write ahead of the prefill runs too)."""
    w = _case("eb", 136, [1, 4], [40, 30], distribution=[0, 0, 0], **_KV[kv])
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    out, pool_after, status = run_gpu(w, q, k, v, pool)
    assert status == 0
    assert np.all(out == 7.0) and torch.equal(pool, pool_after)


def test_host_errors_raise():
    w = _case("he", 134, [1], [10])
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu").to(DEV)
    with pytest.raises(rpa.RpaError):
        rpa.forward(_dev(q), _dev(k), _dev(v), pool, _dev(w.kv_lens), _dev(w.block_tables),
                    _dev(w.query_start_loc), _dev(w.distribution), k_scale=0.5)


# ------------------------------------------------------------- update_cache
@pytest.mark.parametrize("kind", ["bf16", "fp8", "fp8_per_head"])
def test_update_cache_alone_matches_oracle(kind):
    fp8 = kind != "bf16"
    heads = dict(k_scale_heads=[0.03, 0.08], v_scale_heads=[0.2, 0.011]) \
        if kind == "fp8_per_head" else {}
    w = _case("uc", 141, [1, 1, 40, 3], [90, 1, 40, 300], kv_dtype="fp8" if fp8 else "bf16",
              k_scale=0.05 if fp8 else 1.0, v_scale=0.2 if fp8 else 1.0, **heads)
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    p = oracle.make_params(**w.params())
    ref = oracle.update_cache(p, k, v, pool_bytes(pool), w.kv_lens, w.block_tables,
                              w.query_start_loc, w.num_seqs)
    gpool = pool.to(DEV)
    ks = _dev(w.k_scale_heads, torch.float32) if heads else (w.k_scale if fp8 else None)
    vs = _dev(w.v_scale_heads, torch.float32) if heads else (w.v_scale if fp8 else None)
    rpa.update_cache(_dev(k), _dev(v), gpool, _dev(w.kv_lens), _dev(w.block_tables),
                     _dev(w.query_start_loc), _dev(w.distribution), k_scale=ks, v_scale=vs,
                     num_q_heads=w.num_q_heads)
    torch.cuda.synchronize()
    assert np.array_equal(pool_bytes(gpool.cpu()), ref)


def test_fp8_quantisation_sweep_matches_oracle():
    """Every bf16 bit pattern in a wide range, quantised by the page write,
    equals the oracle's E4M3 round-to-nearest-even with saturation."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = bits.astype(np.uint16)
    f = torch.from_numpy(vals.view(np.int16)).view(torch.bfloat16).float()
    keep = torch.isfinite(f) & (f.abs() < 1e30)
    vals = vals[keep.numpy()]
    D, Hkv = 64, 1
    n_tok = -(-len(vals) // (D * Hkv))
    pad = n_tok * D - len(vals)
    allv = np.concatenate([vals, np.zeros(pad, np.uint16)])
    k = torch.from_numpy(allv.view(np.int16)).view(torch.bfloat16).view(n_tok, Hkv, D)
    w = _case("sw", 142, [n_tok], [n_tok], num_q_heads=1, num_kv_heads=1, head_dim=D,
              page_size=64, kv_dtype="fp8", k_scale=0.37, v_scale=1.0)
    pool = w.make_pool("cpu")
    gpool = pool.to(DEV)
    rpa.update_cache(_dev(k), _dev(k), gpool, _dev(w.kv_lens), _dev(w.block_tables),
                     _dev(w.query_start_loc), _dev(w.distribution), k_scale=0.37, v_scale=1.0,
                     num_q_heads=1)
    torch.cuda.synchronize()
    p = oracle.make_params(**w.params())
    ref = oracle.update_cache(p, k, k, pool_bytes(pool), w.kv_lens, w.block_tables,
                              w.query_start_loc, w.num_seqs)
    assert np.array_equal(pool_bytes(gpool.cpu()), ref)


# ------------------------------------------------------- full-size workloads
def _check_subset(w, seqs, pool0, pool, out, q, k, v, sink, sample_tokens_per_seq, nthreads):
    """The listed sequences of a full-size call against the oracle: their
    pages after the call bit for bit, and their outputs (every new token, or
    the first, middle, last and a seeded sample of them)."""
    sub, sub_pool, tmap = w.subset(seqs, pool0)
    p = oracle.make_params(**sub.params())
    cache = oracle.update_cache(p, k[tmap], v[tmap], pool_bytes(sub_pool), sub.kv_lens,
                                sub.block_tables, sub.query_start_loc, sub.num_seqs)
    pages = np.concatenate([w.pages_of(s) for s in seqs]).astype(np.int64)
    got_pages = pool.index_select(0, torch.as_tensor(pages, device=DEV)).cpu()
    assert np.array_equal(pool_bytes(got_pages), cache[:len(pages) * (cache.size // sub.num_pages)])
    if sample_tokens_per_seq is None:
        rows = np.arange(len(tmap))
    else:
        rng = np.random.default_rng(5)
        sqsl = sub.query_start_loc
        rows = []
        for i in range(sub.num_seqs):
            a_, b_ = int(sqsl[i]), int(sqsl[i + 1])
            pick = {a_, b_ - 1, a_ + (b_ - a_) // 2}
            pick |= set(rng.integers(a_, b_, size=sample_tokens_per_seq).tolist())
            rows += sorted(pick)
        rows = np.array(rows)
    ref = oracle.attention_rows(p, q[tmap], cache, sub.kv_lens, sub.block_tables,
                                sub.query_start_loc, sub.num_seqs, rows,
                                None if sink is None else sink.numpy(), nthreads)
    got = out[torch.as_tensor(tmap[rows], device=DEV)].float().cpu().numpy().astype(np.float64)
    return got, ref


def _full_size(name, prefill_seqs=(), sample_tokens_per_seq=None, nthreads=0, batch=32):
    """rpa_forward on the full workload, in the benchmark's launch
    configuration.  Every new-token slot (and nothing else) of the pool must
    change as the page write says; EVERY decode-class sequence is checked
    against the oracle (outputs and pages, in batches of `batch` sequences),
    and the listed prefill sequences on sampled tokens."""
    w = wl.get(name)
    q, k, v = w.make_qkv()
    sink = w.make_sink()
    pool0 = w.make_pool(DEV)
    pool = pool0.clone()
    out = torch.full((w.total_tokens, w.num_q_heads, w.head_dim), 7.0, dtype=torch.bfloat16,
                     device=DEV)
    ws = rpa.alloc_workspace(rpa.make_params(**{a: b for a, b in w.params().items() if a != "kv_fp8"},
                                             kv_fp8=w.kv_dtype == "fp8"), DEV)
    fp8 = w.kv_dtype == "fp8"
    rpa.forward(_dev(q), _dev(k), _dev(v), pool, _dev(w.kv_lens), _dev(w.block_tables),
                _dev(w.query_start_loc), _dev(w.distribution), None if sink is None else _dev(sink),
                softmax_scale=w.softmax_scale, sliding_window=w.sliding_window,
                logits_soft_cap=w.logits_soft_cap, k_scale=w.k_scale if fp8 else None,
                v_scale=w.v_scale if fp8 else None, out=out, workspace=ws)
    assert rpa.get_status(ws) == 0
    torch.cuda.synchronize()
    # every new token's slot, and nothing else, changed as the page write says
    flat0 = pool0.view(w.num_pages * w.page_size, 2 * w.num_kv_heads, w.head_dim)
    flat1 = pool.view(w.num_pages * w.page_size, 2 * w.num_kv_heads, w.head_dim)
    slots = []
    for s in range(w.num_seqs):
        ctx = int(w.kv_lens_valid[s]) - int(w.q_lens[s])
        pos = np.arange(ctx, int(w.kv_lens_valid[s]))
        slots.append(w.block_tables[s * w.pages_per_seq + pos // w.page_size].astype(np.int64)
                     * w.page_size + pos % w.page_size)
    slots = torch.as_tensor(np.concatenate(slots), device=DEV)
    changed = torch.zeros(flat0.shape[0], dtype=torch.bool, device=DEV)
    changed[slots] = True
    assert torch.equal(flat0[~changed], flat1[~changed])
    kd, vd = k.to(DEV), v.to(DEV)
    if fp8:
        kd = (kd.float() / torch.tensor(np.float32(w.k_scale))).to(torch.float8_e4m3fn).view(torch.uint8)
        vd = (vd.float() / torch.tensor(np.float32(w.v_scale))).to(torch.float8_e4m3fn).view(torch.uint8)
    nq = w.num_query_tokens
    assert torch.equal(flat1[slots][:, 0::2], kd[:nq]) and torch.equal(flat1[slots][:, 1::2], vd[:nq])
    assert torch.all(out[nq:] == 7.0)
    del flat0, flat1, changed, kd, vd
    decode_seqs = [s for s in range(w.num_seqs)
                   if s < int(w.distribution[0]) and int(w.q_lens[s]) == 1]
    gots, refs = [], []
    for i in range(0, len(decode_seqs), batch):
        g_, r_ = _check_subset(w, decode_seqs[i:i + batch], pool0, pool, out, q, k, v, sink,
                               None, nthreads)
        gots.append(g_)
        refs.append(r_)
    if prefill_seqs:
        g_, r_ = _check_subset(w, list(prefill_seqs), pool0, pool, out, q, k, v, sink,
                               sample_tokens_per_seq, nthreads)
        gots.append(g_)
        refs.append(r_)
    assert_close(np.concatenate(gots), np.concatenate(refs), name)
    return len(decode_seqs)


def test_full_decode_workload():
    assert _full_size("decode") == 256


def test_full_decode_d256_workload():
    assert _full_size("decode_d256") == 256


def test_full_mixed_workload():
    assert _full_size("mixed", prefill_seqs=[128, 131, 133, 135, 136, 137],
                      sample_tokens_per_seq=6) == 128


def test_full_fp8_workload():
    assert _full_size("fp8", prefill_seqs=[512, 515, 519], sample_tokens_per_seq=8,
                      batch=64) == 512


@pytest.mark.parametrize("name", ["long", "long_w4096", "long_d256"])
def test_full_long_workload(name):
    _full_size(name, prefill_seqs=[0, 1], sample_tokens_per_seq=6)
